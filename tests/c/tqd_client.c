/* A C client of libtqd, using the C ABI alone: build the seeded synthetic
 * model with tqd_create_synthetic, prefill a prompt, run greedy steps on the
 * device with tqd_generate, and print the tokens (the prefill's next token,
 * then one per step) on one line.
 *
 * usage: tqd_client SEED STEPS SCHEDULE N_LAYERS HIDDEN N_HEADS N_KV_HEADS
 *                   HEAD_DIM INTERMEDIATE VOCAB QK_NORM WEIGHT_TYPE
 *                   ROPE_THETA RMS_EPS PROMPT_ID...
 * Exit status 0 on success; 1 with the status name and detail on stderr when
 * a call is refused or fails; 2 on bad usage. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "tqd.h"

static int fail(const char* call, int32_t rc) {
  fprintf(stderr, "%s: %s (%s)\n", call, tqd_status_name(rc), tqd_last_error());
  return 1;
}

int main(int argc, char** argv) {
  const int fixed = 15;
  if (argc < fixed + 1) {
    fprintf(stderr, "usage: %s SEED STEPS SCHEDULE N_LAYERS HIDDEN N_HEADS N_KV_HEADS HEAD_DIM "
                    "INTERMEDIATE VOCAB QK_NORM WEIGHT_TYPE ROPE_THETA RMS_EPS PROMPT_ID...\n", argv[0]);
    return 2;
  }
  const uint64_t seed = strtoull(argv[1], NULL, 10);
  const int steps = atoi(argv[2]);
  const int n_prompt = argc - fixed;
  tqd_config c = {0};
  c.schedule = atoi(argv[3]);
  c.n_layers = atoi(argv[4]);
  c.hidden = atoi(argv[5]);
  c.n_heads = atoi(argv[6]);
  c.n_kv_heads = atoi(argv[7]);
  c.head_dim = atoi(argv[8]);
  c.intermediate = atoi(argv[9]);
  c.vocab = atoi(argv[10]);
  c.qk_norm = atoi(argv[11]);
  c.weight_type = atoi(argv[12]);
  c.rope_theta = strtof(argv[13], NULL);
  c.rms_eps = strtof(argv[14], NULL);
  c.max_seq = n_prompt + steps + 1;
  c.max_batch = 1;
  c.kv_type = TQD_KV_F32;
  if (steps < 1) return 2;
  int32_t* ids = malloc(sizeof(int32_t) * (size_t)n_prompt);
  int32_t* out = malloc(sizeof(int32_t) * (size_t)steps);
  if (!ids || !out) return 2;
  for (int i = 0; i < n_prompt; ++i) ids[i] = (int32_t)atoi(argv[fixed + i]);

  tqd_model* m = NULL;
  int32_t rc = tqd_create_synthetic(&c, seed, NULL, &m);
  if (rc) return fail("tqd_create_synthetic", rc);
  int32_t next = -1;
  if ((rc = tqd_prefill(m, 0, ids, n_prompt, &next))) return fail("tqd_prefill", rc);
  if ((rc = tqd_generate(m, 0, next, steps, out))) return fail("tqd_generate", rc);
  printf("%d", (int)next);
  for (int i = 0; i < steps; ++i) printf(" %d", (int)out[i]);
  printf("\n");
  tqd_destroy(m);
  free(ids);
  free(out);
  return 0;
}
