// Persistent schedule: the bf16-weight kernels (one per head_dim and number
// of q heads per kv head), in their own translation unit so that the two
// formats compile in parallel.
#include "tqd_persist.cuh"

namespace tqd {

const void* persist_fn_bf16(const DevModel& m) {
  const int G = m.nq / m.nkv;
  return m.hd == 128 ? persist_fn_g<kFmtBF16, 128>(G) : persist_fn_g<kFmtBF16, 64>(G);
}

}  // namespace tqd
