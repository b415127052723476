/* The C ABI from plain C99: include/kvc.h compiles as C with every warning
 * an error, and the host-side calls behave as declared without a GPU (the
 * state is host memory that no call below may touch: each either only
 * computes sizes and offsets or fails validation before any launch). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvc.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, #cond); \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  kvc_config cfg;
  kvc_cache* cache = NULL;
  void* raw;
  void* state;
  size_t n, ws;
  void* d_ptr = NULL;
  size_t bytes = 0;
  int32_t slots = -1, pos = -1;
  kvc_evict_params bad;

  CHECK(kvc_version() == KVC_VERSION);
  CHECK(strcmp(kvc_status_string(KVC_OK), "ok") == 0);
  memset(&cfg, 0, sizeof cfg);
  cfg.num_q_heads = 8;
  cfg.num_kv_heads = 2;
  cfg.head_dim = 128;
  cfg.page_size = 16;
  cfg.bits = 4;
  cfg.num_blocks = 8;
  cfg.max_batch = 2;
  cfg.max_blocks_per_seq = 4;
  cfg.bf16_window = 0;
  cfg.codes = KVC_CODES_INT;
  n = kvc_state_bytes(&cfg);
  CHECK(n > 0 && n % 256 == 0);
  raw = malloc(n + 256);
  CHECK(raw != NULL);
  state = (void*)(((uintptr_t)raw + 255) & ~(uintptr_t)255);
  CHECK(kvc_cache_create(&cfg, state, n - 1, &cache) == KVC_ERR_INVALID_ARG);
  CHECK(kvc_cache_create(&cfg, state, n, &cache) == KVC_OK && cache != NULL);
  /* INT4 K codes: num_blocks x Hkv x 16 slots x 64 bytes, at the start */
  CHECK(kvc_cache_buffer(cache, KVC_BUF_K_CODES, &d_ptr, &bytes) == KVC_OK);
  CHECK(d_ptr == state && bytes == (size_t)8 * 2 * 16 * 64);
  CHECK(kvc_cache_buffer(cache, KVC_BUF_COUNT, &d_ptr, &bytes) == KVC_ERR_INVALID_ARG);
  CHECK(kvc_cache_lengths(cache, 0, &slots, &pos) == KVC_OK && slots == 0 && pos == 0);
  ws = kvc_workspace_bytes(cache, 1);
  CHECK(ws > 0);
  CHECK(kvc_prefill_context_workspace_bytes(cache, 1, 8) > 0);
  /* validation before any launch (4 pages of 16 slots hold 68 tokens) */
  CHECK(kvc_quantize_append(cache, 1, 2, 1, state, state, NULL) == KVC_ERR_INVALID_ARG);
  CHECK(kvc_quantize_append(cache, 0, 1, 0, NULL, NULL, NULL) == KVC_OK);
  CHECK(kvc_quantize_append(cache, 0, 1, 4 + 4 * 16 + 1, state, state, NULL) == KVC_ERR_CAPACITY);
  memset(&bad, 0, sizeof bad);
  bad.mode = KVC_EVICT_H2O;
  bad.budget = 10;
  bad.recent = 8; /* budget < 4 + recent */
  CHECK(kvc_h2o_select_evict(cache, 0, 1, &bad, (uint8_t*)state, state, ws, NULL) == KVC_ERR_INVALID_ARG);
  CHECK(kvc_compact_blocks(cache, 0, 1, (const uint8_t*)state, state, ws, NULL) == KVC_ERR_STATE);
  CHECK(kvc_last_launch_count(cache) == 0);
  kvc_cache_destroy(cache);
  free(raw);
  printf("ok\n");
  return 0;
}
