/*
 * fa_gb300.h — C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The library computes exact softmax attention with tiled online softmax, its
 * recompute backward and split-KV decoding, as defined on the web pages
 * "attention_kernels.py" (CMU 15-779 lecture 5), "lab.py" (hs-black
 * flash-attention post) and "flash_attention_numpy.py" (first_principles,
 * flash-attention tier 1).
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer and the stream.  The library
 *    allocates no memory; scratch memory is passed in as `workspace`.
 *  - Pointers are device pointers unless stated otherwise, 16-byte aligned.
 *  - Layout: Q, K, V, O, dO, dQ, dK, dV are contiguous row-major [B, H, N, d]
 *    (batch, head, position, feature); LSE is [B, H, N] float, natural log.
 *  - `scale <= 0` selects the default 1/sqrt(d) ("attention_kernels.py",
 *    section 2, ``_scale``).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is queued asynchronously on it.
 *  - Errors: argument errors return synchronously (FA_ERR_INVALID_ARG,
 *    FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE) and queue nothing.  A failed
 *    launch returns FA_ERR_CUDA.  A kernel that hits its internal wait limit
 *    (it never hangs) records FA_ERR_TIMEOUT, read by fa_get_device_status().
 *  - Supported: d in {64, 128}; N >= 1 (any N: ragged last tiles are masked);
 *    B * H < 2^31, and the forward's B * H * ceil(Nq / 256) work items and the
 *    backward's B * H * ceil(Nk / 128) CTAs below 2^31 as well
 *    (FA_ERR_UNSUPPORTED otherwise); fa_decode: B, H <= 65535.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 3

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, misaligned pointer, bad size */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d not in {64, 128}) */
  FA_ERR_CUDA = 3,        /* a CUDA call or launch failed */
  FA_ERR_TIMEOUT = 4,     /* a kernel gave up waiting (reported by fa_get_device_status) */
  FA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than the *_workspace_size() */
  FA_ERR_BOUNDS = 6       /* a kernel of the bounds-checked build (FA_BOUNDS_CHECK) caught an index
                             outside its buffer and skipped the access (reported by fa_get_device_status) */
} fa_status;

typedef enum fa_dtype { FA_BF16 = 0, FA_F32 = 1 } fa_dtype;

/* Version of this ABI (FA_ABI_VERSION of the built library). */
int fa_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(fa_status s);

/* Bytes of workspace fa_forward and fa_forward_qk need: the persistent grid's
 * work counter, padded to 256 bytes.  The size does not depend on the problem
 * (the arguments are checked only: 0 for B, H, N < 1 or d < 1).  Each call sets
 * the counter to zero on its stream before its kernel starts, so a workspace
 * needs no initialisation; it must not be in use by a call whose GPU work
 * overlaps (two graphs replayed at once need a workspace each). */
size_t fa_forward_workspace_size(int B, int H, int N, int d, int causal);

/*
 * fa_forward — O = softmax(Q K^T * scale [+ causal mask]) V and LSE.
 *
 * Defines: "attention_kernels.py" section 3 ``flash_forward`` (and section 2
 * ``standard_attention`` for the result it must equal): S = Q K^T * scale,
 * online softmax with running max m and denominator l rescaled by
 * exp(m_old - m_new), O = (sum P V) / l, L = m + ln l per query row.
 * With causal != 0, key j is visible to query i iff j <= i (q_start = 0).
 *
 *  q, k, v   [B, H, N, d] bf16, read only.
 *  o         [B, H, N, d], written; o_dtype FA_BF16 or FA_F32.
 *  lse       [B, H, N] float, written (natural log).
 *  precise   0: P is rounded to bf16 before the P V product (standard).
 *            1: P enters P V as a bf16 high part plus a bf16 residual (two
 *               tensor-core products), for fp32-grade outputs.
 *  workspace device scratch of >= fa_forward_workspace_size() bytes, 16-byte
 *            aligned, owned by the caller (FA_ERR_WORKSPACE if missing or small).
 * Returns FA_OK when the work is queued.
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype, float* lse, int B,
                     int H, int N, int d, float scale, int causal, int precise, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * fa_forward_qk — fa_forward with Nq queries against Nk keys and a query offset.
 *
 * Defines: "attention_kernels.py" section 3 ``flash_forward`` with its ``q_start``
 * (section 2 ``_mask``): query row i sits at absolute position q_start + i and,
 * with causal != 0, sees key j iff j <= q_start + i.  Without causal every query
 * sees every key (cross-attention when Nq != Nk).  Covers chunked prefill
 * (q_start = Nk - Nq) and multi-token decoding with a causal mask.
 *
 *  q   [B, H, Nq, d] bf16;  k, v  [B, H, Nk, d] bf16.
 *  o   [B, H, Nq, d] in o_dtype, written;  lse  [B, H, Nq] float, written.
 *  Nq, Nk >= 1;  q_start >= 0 (every query then sees key 0) and q_start + Nq
 *  must fit in int: otherwise FA_ERR_INVALID_ARG.  Workspace as for fa_forward.
 *  fa_forward(..., N, ...) is fa_forward_qk(..., Nq = Nk = N, q_start = 0, ...).
 */
fa_status fa_forward_qk(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype, float* lse, int B,
                        int H, int Nq, int Nk, int q_start, int d, float scale, int causal, int precise,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace fa_backward needs (pass Nq for fa_backward_qk): 64 per query row over N rounded up to a
 * multiple of 64 (per row, -LSE/scale and -rowsum(dO * O), each as three bf16
 * terms, laid out as tensor-core operand tiles); with grad_dtype FA_BF16 also
 * the fp32 accumulator of dQ (4 * N * d bytes per (batch, head), after the
 * tiles at a 256-byte boundary).  0 for an invalid argument. */
size_t fa_backward_workspace_size(int B, int H, int N, int d, fa_dtype grad_dtype);

/*
 * fa_backward — dQ, dK, dV of loss = sum(O * dO) by recomputing P from LSE.
 *
 * Defines: "attention_kernels.py" section 4 ``flash_backward``:
 * D = rowsum(dO * O); per key tile and query tile P = exp(S - L),
 * dV += P^T dO, dP = dO V^T, dS = P * (dP - D), dQ += dS K * scale,
 * dK += dS^T Q * scale.  The N x N matrices are never stored.
 *
 *  q, k, v, dout  [B, H, N, d] bf16; o [B, H, N, d] in o_dtype (the forward's
 *                 output); lse [B, H, N] float (the forward's LSE).
 *  dq, dk, dv     [B, H, N, d] in grad_dtype, written.  Every product
 *                 accumulates in fp32; FA_BF16 rounds the final gradients to
 *                 bf16 (dQ is accumulated in the workspace and converted by a
 *                 second kernel), FA_F32 writes them as they are (dQ is zeroed
 *                 and accumulated in place).  Another grad_dtype is
 *                 FA_ERR_INVALID_ARG.
 *  workspace      device scratch of >= fa_backward_workspace_size(..., grad_dtype) bytes.
 * The causal flag and scale must match the forward call.
 */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, fa_dtype o_dtype,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, fa_dtype grad_dtype, int B,
                      int H, int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * fa_backward_qk — fa_backward with Nq queries against Nk keys and a query offset.
 *
 * Defines: the gradient of fa_forward_qk's result ("attention_kernels.py"
 * section 4 ``flash_backward``, whose recompute of P uses the same mask as the
 * forward).  Keys no query sees (positions after q_start + Nq - 1 under causal)
 * get zero dK and dV.
 *
 *  q, dout, o  [B, H, Nq, d];  lse [B, H, Nq];  k, v [B, H, Nk, d].
 *  dq [B, H, Nq, d];  dk, dv [B, H, Nk, d]; in grad_dtype, written (as for fa_backward).
 *  workspace   >= fa_backward_workspace_size(B, H, Nq, d, grad_dtype) bytes.
 * Lengths and offset as for fa_forward_qk; they, causal and scale must match
 * the forward call.
 */
fa_status fa_backward_qk(const void* q, const void* k, const void* v, const void* o, fa_dtype o_dtype,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, fa_dtype grad_dtype, int B,
                         int H, int Nq, int Nk, int q_start, int d, float scale, int causal, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Bytes of workspace fa_decode needs: per-segment states (B * H * n_split * (d + 2)
 * floats) and one arrival counter per (batch, head), each part padded to 256
 * bytes.  0 for an argument < 1, or for a size beyond 2^62 bytes (the counts are
 * checked before they are multiplied, so the size never wraps around). */
size_t fa_decode_workspace_size(int B, int H, int d, int n_split);

/*
 * fa_decode — one query per (batch, head) against L keys, split-KV.
 *
 * Defines: "attention_kernels.py" section 5 ``flash_decode``: the L keys are
 * split into n_split segments with bounds round(L * s / n_split) (ties to
 * even), each segment yields its softmax state (m, l, o) (section 1
 * ``SoftmaxState``), and the states are merged left to right with
 * ``merge_states``; O = o / l.  No causal mask (the query sees every key).
 * Segments may be empty (n_split > L) and then contribute the identity state.
 *
 *  q          [B, H, 1, d] bf16;  k, v  [B, H, L, d] bf16.
 *  o          [B, H, 1, d] float, written;  lse  [B, H] float, written.
 *  partials   optional [B, H, n_split, d + 2] float: per segment (m, l, o[d])
 *             with m in natural-log units; NULL to skip.
 *  workspace  device scratch of >= fa_decode_workspace_size() bytes; the call
 *             clears the counters it holds on `stream` before the kernel runs.
 *  n_split    >= 1 (n_split < 1 is FA_ERR_INVALID_ARG, as the page raises).
 * B, H > 65535, n_split > 2^30, or a workspace size beyond 2^62 bytes is
 * FA_ERR_UNSUPPORTED; a workspace smaller than fa_decode_workspace_size() is
 * FA_ERR_WORKSPACE.
 */
fa_status fa_decode(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H, int L, int d,
                    float scale, int n_split, float* partials, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * fa_decode_auto_split — a split count for fa_decode: B * H heads of L keys on
 * the current device.  Returns n_split >= 1, or 0 if an argument is < 1 or the
 * device cannot be queried.
 *
 * The pages leave n_split to the caller ("attention_kernels.py" section 5).  The
 * rule, from measurements of fa_decode on GB300 over n_split in 1..256: about
 * four CTAs per SM in all (ceil(4 * SMs / (B * H)) splits), at least 8, and no
 * segment shorter than 512 keys (at most L / 512 splits, at least 1).  Size the
 * workspace with the same n_split.
 */
int fa_decode_auto_split(int B, int H, int L);

/* Size in bytes of the fixed scratch array behind fa_decode_noalloc. */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * fa_decode_noalloc — fa_decode for callers that can neither pass a workspace
 * nor allocate device memory.  The pages have no counterpart: this is a
 * library convenience, not part of the method.
 *
 * Who needs it: code that may not call cudaMalloc, for example a plugin or
 * callback run by a framework that owns all device memory and hands it no
 * workspace, or a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable.
 *
 * Same arguments, results and errors as fa_decode, minus the workspace.  The
 * scratch memory is one fixed array of FA_DECODE_NOALLOC_SCRATCH_BYTES
 * (16 MiB) in device memory, held by every GPU that loads the library until
 * the process exits.  A call needs fa_decode_workspace_size(B, H, d, n_split)
 * bytes of it and returns FA_ERR_WORKSPACE, queueing nothing, when that is
 * larger than FA_DECODE_NOALLOC_SCRATCH_BYTES.  Nothing is allocated: no
 * cudaMalloc, no cudaFree, no allocating library call.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array and each leaves
 * its contents behind (the call clears the counters it needs on `stream`), so
 * calls whose GPU work overlaps, on different streams or from different host
 * threads, race with each other; serialise them.
 */
fa_status fa_decode_noalloc(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H, int L,
                            int d, float scale, int n_split, float* partials, void* stream);

/*
 * fa_get_device_status — synchronises `stream`, reads and clears the kernels'
 * device status words.  Returns FA_ERR_TIMEOUT if any kernel gave up on a
 * wait since the last call, FA_ERR_BOUNDS if the bounds-checked build caught
 * an index outside its buffer, FA_ERR_CUDA if the CUDA calls fail, else FA_OK.
 */
fa_status fa_get_device_status(void* stream);

/* fa_device_status — the same call as fa_get_device_status (earlier name, kept). */
fa_status fa_device_status(void* stream);

/* Bytes of workspace fa_forward_keymajor needs: the running O (fp32), maximum and
 * sum of every query row. */
size_t fa_forward_keymajor_workspace_size(int B, int H, int N, int d);

/*
 * fa_forward_keymajor — the forward in the first algorithm's loop order, for
 * comparison with fa_forward.  Same result as fa_forward (O and LSE), by a
 * different schedule: key tiles outer, query tiles inner, and the running output,
 * maximum and sum of every query row kept in the workspace and repaired at every
 * visit, O renormalised each time.
 *
 * Defines: "flash_attention_numpy.py" ``flash_attention_tier1`` (key blocks
 * outer, query blocks inner; r' = e^(m - m') r + e^(m~ - m') r~,
 * O = (e^(m - m') r / r') O + e^(m~ - m') (p~ V_j) / r'), with the scale and the
 * causal skip and mask of "attention_kernels.py" section 3.  Blocks are 128 x 128.
 * One CTA per (batch, head) and no overlap between the steps of a visit: it
 * shows the loop order, and is much slower than fa_forward.
 *
 * Arguments as for fa_forward (no precise mode), plus a workspace of
 * >= fa_forward_keymajor_workspace_size() bytes, 16-byte aligned.
 */
fa_status fa_forward_keymajor(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype, float* lse,
                              int B, int H, int N, int d, float scale, int causal, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * fa_merge_states — combines two attention results over disjoint key sets.
 *
 * Defines: "attention_kernels.py" section 1 ``merge_states``: softmax states
 * (m, l, o) of two runs of scores merge as m = max(m_a, m_b),
 * l = l_a e^(m_a - m) + l_b e^(m_b - m), o likewise.  A normalised result
 * (O, LSE) is the state (LSE, 1, O), so per row, with m = max(LSE_a, LSE_b) and
 * w = e^(LSE - m):  LSE = m + ln(w_a + w_b),  O = (w_a O_a + w_b O_b) / (w_a + w_b).
 * LSE = -inf marks an empty run, the identity; two empty runs give O = 0 and
 * LSE = -inf.  Typical use: attention over keys held in two pieces (two
 * fa_forward_qk calls without causality, or two fa_decode calls), merged into
 * the result over all keys.
 *
 *  o_a, o_b, o      rows x d, contiguous per row, in o_dtype (FA_F32 or
 *                   FA_BF16); 16-byte aligned.  o may be o_a or o_b.
 *  lse_a, lse_b, lse  rows floats (natural log); lse may be lse_a or lse_b.
 *  rows >= 0 (0 queues nothing);  d a multiple of 4 in [4, 4096].
 * Returns FA_OK when queued; FA_ERR_INVALID_ARG for null or misaligned
 * pointers or bad sizes.
 */
fa_status fa_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o,
                          float* lse, fa_dtype o_dtype, long long rows, int d, void* stream);

/*
 * fa_set_stats — counters of the pages' ``stats`` dictionary, for debugging and
 * tests.
 *
 * Defines: "attention_kernels.py" section 3 ``flash_forward`` (counters
 * "tiles", "skipped", "rescales") and section 4 ``flash_backward``
 * ("dq_atomic_adds").  While a buffer is set, every fa_forward and fa_backward
 * call made from the calling host thread adds into it.  `counters` is device
 * memory: 4 unsigned 64-bit words, zeroed by the caller, owned by the caller.
 *   [0] tiles           (query tile of 128 rows, key tile of 128) pairs the
 *                       forward computed; query tiles that start at or past N
 *                       do not count.
 *   [1] skipped         such pairs the forward skipped under causality (the key
 *                       tile starts after the query tile's last row).
 *   [2] rescales        (query row, computed key tile) pairs in which the row's
 *                       running maximum score grew from a finite value; rows at
 *                       or past N do not count.
 *   [3] dq_atomic_adds  dQ elements the backward added: per computed (query
 *                       block of 64 rows, key tile of 128) pair, its rows (fewer
 *                       in a last, partial block) times d.
 * Summed over batch and heads, these equal the page's counts for blocks
 * Br = Bc = 128 (forward) and Br = 64, Bc = 128 (backward) times B * H, since the
 * page counts each block pair once for all heads; "rescales" equals the page's
 * count directly (the page sums it over all rows).  The kernels add each CTA's
 * counts once, at its end, so counting costs next to nothing.  NULL (the
 * default) stops counting.  Returns FA_OK; FA_ERR_INVALID_ARG if `counters` is
 * not 8-byte aligned.
 */
fa_status fa_set_stats(unsigned long long* counters);

/*
 * fa_debug_wait_timeout — test hook for the failure path: queues one CTA that
 * waits on a barrier nothing completes, with a limit of `limit_ns`
 * nanoseconds.  The kernel returns on its own; the next fa_get_device_status()
 * must report FA_ERR_TIMEOUT.
 */
fa_status fa_debug_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * fa_debug_abort_next_call — test hook for the failure path of the real kernels:
 * the next fa_forward, fa_forward_qk, fa_backward or fa_backward_qk call made
 * from the calling host thread runs its kernel as if a wait on its own pipeline
 * had timed out at the start (the MMA-issuing role raises the CTA's abort flag and
 * records the timeout).  Every other role then leaves its loop through its own
 * bounded wait, the copies and products already issued are waited for, tensor
 * memory is freed and the kernel returns; that call's outputs are undefined and
 * the next fa_get_device_status() reports FA_ERR_TIMEOUT.  The flag is taken by
 * that one call.  Returns FA_OK.
 */
fa_status fa_debug_abort_next_call(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
