// Internal launch interface shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_gb300.h"

namespace fa {


struct ForwardArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [B*H, Nq or Nk, d] bf16, box {64, 128, 1}, 128B swizzle
  void* o;                       // [B, H, Nq, d] bf16 or fp32
  float* lse;                    // [B, H, Nq] natural-log log-sum-exp
  int B, H, Nq, Nk, d;
  int q_start;                   // absolute position of query row 0 (causal: key j visible iff j <= q_start + i)
  float scale_log2;              // scale * log2(e)
  int causal;
  int o_f32;                     // 1: O is fp32, 0: bf16
  int precise;                   // 1: P enters PV as a bf16 hi + lo pair (two MMAs)
  unsigned* sched;               // work items claimed so far: a counter in the caller's workspace, zeroed
                                 // on the stream before the launch
  int head_group;                // heads interleaved in the work order (set by the API, see head_group_for)
  unsigned long long* stats;     // optional counters [tiles, skipped, rescales, dq adds]; null: none
  int debug_abort;               // failure-path test: the kernel aborts as after a timed-out wait
};

struct BackwardArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // 3-D maps over [B*H, Nq or Nk, d] bf16; Q, dO boxes of 64 rows, K, V of 128
  CUtensorMap tm_dk, tm_dv;             // 3-D maps over dK, dV [B*H, Nk, d], boxes of 128 rows x 128 bytes
                                        // ({32, 128, 1} fp32 or {64, 128, 1} bf16), 128B swizzle
  const void* o;                        // [B, H, Nq, d] bf16 or fp32
  const void* dout;                     // [B, H, Nq, d] bf16
  const float* lse;                     // [B, H, Nq]
  float* dq;                            // [B, H, Nq, d] fp32 accumulator (zeroed by the preprocess): the output
                                        // itself for fp32 gradients, workspace for bf16 ones
  void* dq_out;                         // [B, H, Nq, d] dQ output in the gradient type
  void* dk;                             // [B, H, Nk, d] in the gradient type
  void* dv;                             // [B, H, Nk, d] in the gradient type
  int grad_bf16;                        // gradients written as bf16 (else fp32)
  uint8_t* bias;                        // workspace [B*H, n_pad / 64] blocks of 4 KB: per 64-query block the
                                        // bias tiles -LSE/scale and -rowsum(dO * O) (-inf and 0 past Nq)
  int n_pad;                            // Nq rounded up to a multiple of 64
  int B, H, Nq, Nk, d;
  int q_start;                          // absolute position of query row 0, as in the forward
  float scale;                          // softmax scale
  float scale_log2;                     // scale * log2(e)
  int causal;
  int o_f32;
  int head_group;                       // heads interleaved in the grid order (set by the API, see head_group_for)
  unsigned long long* stats;            // optional counters [tiles, skipped, rescales, dq adds]; null: none
  int debug_abort;                      // failure-path test: the kernel aborts as after a timed-out wait
};

// Heads whose blocks are interleaved in the work order.  Under causality a block's
// work grows with its position, and interleaving heads lets the longest blocks of
// several heads start first, which shortens the tail; the interleaved heads' K and V
// (forward) or Q, dO and dQ (backward) must then share L2.  When every head's data
// fits a 64 MB budget together, all heads form one group: the whole grid then runs
// longest blocks first.  Otherwise a group holds as many heads as fit the budget, at
// most 8, and the heads are split into groups of equal size (a small last group
// would start its longest blocks late).  Without causality every block has the same
// work and one head at a time keeps the most in L2.
inline int head_group_for(int causal, long long bytes_per_head, int n_bh) {
  if (!causal || n_bh < 1) return 1;
  constexpr long long kBudget = 64ll << 20;
  if (bytes_per_head > 0 && static_cast<long long>(n_bh) <= kBudget / bytes_per_head) return n_bh;
  long long fit = kBudget / (bytes_per_head > 0 ? bytes_per_head : 1);
  fit = fit < 1 ? 1 : (fit > 8 ? 8 : fit);
  const long long groups = (n_bh + fit - 1) / fit;
  return static_cast<int>((n_bh + groups - 1) / groups);
}

struct DecodeArgs {
  const void* q;         // [B, H, 1, d] bf16
  const void* k;         // [B, H, L, d] bf16
  const void* v;         // [B, H, L, d] bf16
  float* o;              // [B, H, 1, d]
  float* lse;            // [B, H, 1]
  float* partials;       // optional [B, H, n_split, d + 2] (m, l, o) in natural-log units, or null
  float* ws_partials;    // [B, H, n_split, d + 2] (m in log2 units)
  unsigned* ws_counters; // [B, H] arrival counters, zero on entry; left at zero on exit
  int B, H, L, d, n_split;
  float scale_log2;
};

// The first algorithm's loop order (fa_fwd_keymajor.cu): square case only.
struct KeyMajorArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [B*H, N, d] bf16, box {64, 128, 1}, 128B swizzle
  void* o;                       // [B, H, N, d] bf16 or fp32
  float* lse;                    // [B, H, N]
  float* ws_o;                   // workspace: running O [B*H, N, d] fp32
  float* ws_m;                   // running max (log2 units) [B*H, N]
  float* ws_r;                   // running sum [B*H, N]
  int B, H, N, d;
  float scale_log2;
  int causal;
  int o_f32;
};

// Each returns a cudaError_t from the launch (cudaSuccess when queued).
cudaError_t launch_forward(const ForwardArgs& a, cudaStream_t stream);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_forward_keymajor(const KeyMajorArgs& a, cudaStream_t stream);

// Merge of two (O, LSE) results over disjoint key sets (fa_merge.cu); o_f32: O is
// fp32, else bf16.  O rows of d elements, d a multiple of 4.
cudaError_t read_clear_merge_status(unsigned* out, cudaStream_t stream);
cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o, float* lse,
                         long long rows, int d, int o_f32, cudaStream_t stream);

// Argument checks of fa_decode, shared with fa_decode_noalloc (fa_api.cu): the
// workspace the call needs against `workspace_bytes`; no CUDA call.
fa_status check_decode_args(const void* q, const void* k, const void* v, const float* o, const float* lse, int B,
                            int H, int L, int d, int n_split, size_t workspace_bytes);

// Split count of the decode path for B*H heads of L keys on `sms` SMs.
int decode_auto_split(int BH, int L, int sms);

// Device status words, one per kernel file: read and cleared on `stream`.
cudaError_t read_clear_forward_status(unsigned* out, cudaStream_t stream);
cudaError_t read_clear_backward_status(unsigned* out, cudaStream_t stream);
cudaError_t read_clear_decode_status(unsigned* out, cudaStream_t stream);
cudaError_t read_clear_keymajor_status(unsigned* out, cudaStream_t stream);

// Test hook: one CTA waits on an mbarrier that nothing completes, with the
// given limit in nanoseconds; it must come back with the timeout bit set.
cudaError_t launch_wait_timeout_probe(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace fa
