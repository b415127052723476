// Prefill: the causal attention of a fresh prompt over itself and the H2O
// scores it gives (Technical Report section 3.4: a token's score is the sum,
// over the query rows of the attention matrix, of its probabilities; the
// eviction-and-reuse survey page's section 3.3: its cumulative attention from
// the later tokens).  The prompt attends with its exact bf16 values; its
// tokens are stored quantised (or in the bf16 window) by the append that runs
// first, and the scores initialise the decode steps' H2O accumulation.
//
// Two kernels, both on the fifth-generation tensor cores (kvc_prefill_tc.cu):
// the forward (the bf16 output and each query row's (max, sum)), then the
// scores, which recompute S = Q K^T (the same exact products) per key tile,
// turn it into probabilities with the forward's row statistics and sum them
// over the query rows of the group's query heads into the tokens' score
// slots (sinks, pool or bf16 window).
//
// A prompt over sequences that already hold context (kvc_prefill_context)
// attends to the compressed cache instead (kvc_context.cu).
#include "kvc_internal.h"

namespace kvc {

cudaError_t launch_prefill(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q, const uint16_t* k,
                           const uint16_t* v, uint16_t* out, float* stats, float qk_scale_log2, bool scores,
                           cudaStream_t st, cudaEvent_t trace_start, cudaEvent_t trace_stop) {
  cudaError_t e = trace_start ? cudaEventRecord(trace_start, st) : cudaSuccess;
  if (e != cudaSuccess) return e;
  e = launch_prefill_fwd_tc(s, batch, n, q, k, v, out, stats, qk_scale_log2, st);
  if (e == cudaSuccess && trace_stop) e = cudaEventRecord(trace_stop, st);
  if (e != cudaSuccess || !scores) return e;
  return launch_prefill_scores_tc(s, seq_begin, batch, n, q, k, stats, qk_scale_log2, st);
}

}  // namespace kvc
