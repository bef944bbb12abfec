// Persistent schedule, Q8_0 kernels and the host side: shared memory size,
// support check, occupancy and the cooperative launch.  The device code is in
// tqd_persist.cuh; the bf16 kernels are compiled in tqd_persist_bf16.cu.
#include "tqd_persist.cuh"

namespace tqd {

const void* persist_fn_bf16(const DevModel& m);  // tqd_persist_bf16.cu

namespace {

const void* persist_fn(const DevModel& m) {
  const int G = m.nq / m.nkv;
  if (m.wtype == kFmtQ8) return m.hd == 128 ? persist_fn_g<kFmtQ8, 128>(G) : persist_fn_g<kFmtQ8, 64>(G);
  return persist_fn_bf16(m);
}

}  // namespace

size_t persistent_smem_bytes(const DevModel& m) { return playout(m).total; }

bool persistent_supported(const DevModel& m) {
  const int G = m.nq / m.nkv;
  // the down projection's column pieces: 16-byte aligned runs that fit a slot
  const bool dcol_ok = m.wtype == kFmtQ8 ? (m.H % 16 == 0 && a16(2u * m.H) + 32u * m.H <= kSlotBytes)
                                         : (m.H % 8 == 0 && 2u * m.H <= kSlotBytes);
  return G >= 1 && G <= 4 && (m.hd == 64 || m.hd == 128) && m.H <= kMaxGain * kCT &&
         dcol_ok && m.I % 32 == 0;
}

int persistent_blocks_per_sm(const DevModel& m) {
  if (!persistent_supported(m)) return 0;
  const void* fn = persist_fn(m);
  const size_t smem = persistent_smem_bytes(m);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_persistent(const DevModel& m, const DevSeq& s, int n_steps, int full_from,
                              int blocks, cudaStream_t st) {
  void* params[] = {const_cast<DevModel*>(&m), const_cast<DevSeq*>(&s), &n_steps, &full_from};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = persistent_smem_bytes(m);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, persist_fn(m), params);
}

}  // namespace tqd
