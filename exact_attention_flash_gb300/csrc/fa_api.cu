// C ABI: argument checks, TMA descriptor set-up and launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_gb300.h"
#include "internal.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [B*H, N, d] bf16 viewed as a 3-D tensor (d innermost), tiles of `box_rows` rows x
// 64 features (128 bytes, the swizzle width); rows past N read as zero.
fa_status make_row_tile_map(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// dK or dV [B*H, N, d] as a 3-D tensor, tiles of 128 rows x 128 bytes (32 fp32 or 64
// bf16 features) with the 128-byte swizzle: the backward stores each key tile's
// gradients with bulk tensor stores; rows past N are dropped.
fa_status make_grad_store_map(CUtensorMap* m, void* ptr, int BH, int N, int d, bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  const cuuint64_t esize = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esize, static_cast<cuuint64_t>(N) * d * esize};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), 128, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims,
                         strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr long long kMaxCount = 0x7FFFFFFFLL;

fa_status check_common(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  // Heads, work items and CTAs are counted with 32-bit integers: B*H (and each
  // launch's item or CTA count, checked where it is known) must stay below 2^31.
  if (static_cast<long long>(B) * H > kMaxCount) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Query and key lengths and the query offset: Nq, Nk >= 1, q_start >= 0, and the
// last query position q_start + Nq - 1 inside int.
fa_status check_lengths(int B, int H, int Nq, int Nk, int q_start, int d) {
  fa_status st = check_common(B, H, Nq, d);
  if (st != FA_OK) return st;
  if (Nk < 1 || q_start < 0 || static_cast<long long>(q_start) + Nq > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

float resolve_scale(float scale, int d) { return scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d)); }

constexpr float kLog2e = 1.4426950408889634f;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Backward workspace: the bias tiles, then (bf16 gradients) the fp32 dQ accumulator.
size_t backward_bias_bytes(int B, int H, int N) {
  return static_cast<size_t>(B) * H * round_up(static_cast<size_t>(N), 64) * 64;
}

// Counters set by fa_set_stats for the calling host thread's calls (null: none).
thread_local unsigned long long* t_stats = nullptr;

// Set by fa_debug_abort_next_call: the calling host thread's next forward or
// backward call aborts on purpose; taken (and cleared) by that one call.
thread_local bool t_abort_next = false;

int take_debug_abort() {
  const bool v = t_abort_next;
  t_abort_next = false;
  return v ? 1 : 0;
}

// The forward's workspace: one 32-bit work counter, padded.
constexpr size_t kForwardWorkspaceBytes = 256;

}  // namespace

namespace fa {

// Argument checks shared by fa_decode and fa_decode_noalloc, in one place so that
// the two entry points cannot drift apart: pointers, sizes, and the workspace the
// call needs, fa_decode_workspace_size(B, H, d, n_split), against `workspace_bytes`
// (the caller's workspace, or the fixed scratch array).  No CUDA call.
fa_status check_decode_args(const void* q, const void* k, const void* v, const float* o, const float* lse, int B,
                            int H, int L, int d, int n_split, size_t workspace_bytes) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FA_ERR_INVALID_ARG;
  if (n_split < 1 || L < 1 || B < 1 || H < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B > 65535 || H > 65535 || n_split > (1 << 30)) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_decode_workspace_size(B, H, d, n_split);
  if (need == 0) return FA_ERR_UNSUPPORTED;  // beyond any device's memory
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  return FA_OK;
}

}  // namespace fa

extern "C" {

int fa_abi_version(void) { return FA_ABI_VERSION; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_BOUNDS: return "index outside its buffer (bounds-checked build)";
  }
  return "unknown status";
}

size_t fa_forward_workspace_size(int B, int H, int N, int d, int causal) {
  (void)causal;
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return kForwardWorkspaceBytes;
}

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype, float* lse, int B,
                     int H, int N, int d, float scale, int causal, int precise, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return fa_forward_qk(q, k, v, o, o_dtype, lse, B, H, N, N, 0, d, scale, causal, precise, workspace,
                       workspace_bytes, stream);
}

fa_status fa_forward_qk(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype, float* lse, int B,
                        int H, int Nq, int Nk, int q_start, int d, float scale, int causal, int precise,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (o_dtype != FA_BF16 && o_dtype != FA_F32) return FA_ERR_INVALID_ARG;
  fa_status st = check_lengths(B, H, Nq, Nk, q_start, d);
  if (st != FA_OK) return st;
  if (static_cast<long long>(B) * H * ((Nq + 255) / 256) > kMaxCount) return FA_ERR_UNSUPPORTED;  // work items
  if (!workspace || !aligned16(workspace) || workspace_bytes < kForwardWorkspaceBytes) return FA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fa::ForwardArgs a{};
  const int BH = B * H;
  if ((st = make_row_tile_map(&a.tm_q, q, BH, Nq, d)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_k, k, BH, Nk, d)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_v, v, BH, Nk, d)) != FA_OK) return st;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.q_start = q_start;
  a.d = d;
  a.scale_log2 = resolve_scale(scale, d) * kLog2e;
  a.causal = causal ? 1 : 0;
  a.head_group = fa::head_group_for(a.causal, 2ll * Nk * d * 2, B * H);  // K and V of a head, bf16
  a.o_f32 = (o_dtype == FA_F32) ? 1 : 0;
  a.precise = precise ? 1 : 0;
  a.stats = t_stats;
  a.debug_abort = take_debug_abort();
  // The persistent grid claims its work items from this counter: zero it first,
  // in stream order, so that the workspace needs no initialisation by the caller.
  a.sched = static_cast<unsigned*>(workspace);
  if (cudaMemsetAsync(a.sched, 0, sizeof(unsigned), s) != cudaSuccess) return FA_ERR_CUDA;
  return fa::launch_forward(a, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Per query row over [B*H, N rounded up to 64]: two 32-byte rows of the bias tiles
// (-LSE/scale and -D as three bf16 terms each); for bf16 gradients then, at a 256-byte
// boundary, the fp32 dQ accumulator [B, H, N, d].
size_t fa_backward_workspace_size(int B, int H, int N, int d, fa_dtype grad_dtype) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  if (grad_dtype == FA_F32) return backward_bias_bytes(B, H, N);
  if (grad_dtype != FA_BF16) return 0;
  return round_up(backward_bias_bytes(B, H, N), 256) + static_cast<size_t>(B) * H * N * d * sizeof(float);
}

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, fa_dtype o_dtype,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, fa_dtype grad_dtype, int B,
                      int H, int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return fa_backward_qk(q, k, v, o, o_dtype, lse, dout, dq, dk, dv, grad_dtype, B, H, N, N, 0, d, scale, causal,
                        workspace, workspace_bytes, stream);
}

fa_status fa_backward_qk(const void* q, const void* k, const void* v, const void* o, fa_dtype o_dtype,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, fa_dtype grad_dtype, int B,
                         int H, int Nq, int Nk, int q_start, int d, float scale, int causal, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if (o_dtype != FA_BF16 && o_dtype != FA_F32) return FA_ERR_INVALID_ARG;
  if (grad_dtype != FA_BF16 && grad_dtype != FA_F32) return FA_ERR_INVALID_ARG;
  fa_status st = check_lengths(B, H, Nq, Nk, q_start, d);
  if (st != FA_OK) return st;
  // one CTA per (128-key tile, head); the preprocess takes 256 / (d / 8) rows per block
  if (static_cast<long long>(B) * H * ((Nk + 127) / 128) > kMaxCount ||
      static_cast<long long>(B) * H * ((Nq + 63) / 64 * 64) / (256 / (d / 8)) > kMaxCount)
    return FA_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < fa_backward_workspace_size(B, H, Nq, d, grad_dtype))
    return FA_ERR_WORKSPACE;
  const bool grad_bf16 = grad_dtype == FA_BF16;
  fa::BackwardArgs a{};
  const int BH = B * H;
  if ((st = make_row_tile_map(&a.tm_q, q, BH, Nq, d, 64)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_k, k, BH, Nk, d, 128)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_v, v, BH, Nk, d, 128)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_do, dout, BH, Nq, d, 64)) != FA_OK) return st;
  if ((st = make_grad_store_map(&a.tm_dk, dk, BH, Nk, d, grad_bf16)) != FA_OK) return st;
  if ((st = make_grad_store_map(&a.tm_dv, dv, BH, Nk, d, grad_bf16)) != FA_OK) return st;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = grad_bf16 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              round_up(backward_bias_bytes(B, H, Nq), 256))
                   : static_cast<float*>(dq);
  a.dq_out = dq;
  a.dk = dk;
  a.dv = dv;
  a.grad_bf16 = grad_bf16 ? 1 : 0;
  a.n_pad = static_cast<int>(round_up(static_cast<size_t>(Nq), 64));
  a.bias = static_cast<uint8_t*>(workspace);
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.q_start = q_start;
  a.d = d;
  a.scale = resolve_scale(scale, d);
  a.scale_log2 = a.scale * kLog2e;
  a.causal = causal ? 1 : 0;
  a.head_group = fa::head_group_for(a.causal, 2ll * Nq * d * 2 + static_cast<long long>(Nq) * d * 4, B * H);  // Q, dO, dQ
  a.o_f32 = (o_dtype == FA_F32) ? 1 : 0;
  a.stats = t_stats;
  a.debug_abort = take_debug_abort();
  const cudaError_t e = fa::launch_backward(a, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Every count is checked before it is multiplied: the segment states take
// B * H * n_split * (d + 2) floats, and a product that would pass 2^62 bytes
// (far beyond any device) is reported as 0, never wrapped around.
size_t fa_decode_workspace_size(int B, int H, int d, int n_split) {
  if (B < 1 || H < 1 || n_split < 1 || d < 1) return 0;
  constexpr size_t kLimit = size_t(1) << 62;
  const size_t heads = static_cast<size_t>(B) * static_cast<size_t>(H);  // < 2^62
  const size_t state_bytes = (static_cast<size_t>(d) + 2) * sizeof(float);
  if (heads > kLimit / static_cast<size_t>(n_split) || heads * n_split > kLimit / state_bytes) return 0;
  const size_t counters = round_up(heads * sizeof(unsigned), 256);
  const size_t partials = heads * n_split * state_bytes;
  return counters + round_up(partials, 256);
}

fa_status fa_decode(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H, int L, int d,
                    float scale, int n_split, float* partials, void* workspace, size_t workspace_bytes,
                    void* stream) {
  fa_status st = fa::check_decode_args(q, k, v, o, lse, B, H, L, d, n_split, workspace_bytes);
  if (st != FA_OK) return st;
  if (!workspace || !aligned16(workspace)) return FA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t counter_bytes = round_up(static_cast<size_t>(B) * H * sizeof(unsigned), 256);
  fa::DecodeArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.partials = partials;
  a.ws_counters = static_cast<unsigned*>(workspace);
  a.ws_partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + counter_bytes);
  a.B = B;
  a.H = H;
  a.L = L;
  a.d = d;
  a.n_split = n_split;
  a.scale_log2 = resolve_scale(scale, d) * kLog2e;
  if (cudaMemsetAsync(a.ws_counters, 0, static_cast<size_t>(B) * H * sizeof(unsigned), s) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa::launch_decode(a, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_forward_keymajor_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return round_up(rows * d * sizeof(float), 256) + 2 * round_up(rows * sizeof(float), 256);
}

fa_status fa_forward_keymajor(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype, float* lse,
                              int B, int H, int N, int d, float scale, int causal, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (o_dtype != FA_BF16 && o_dtype != FA_F32) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, N, d);
  if (st != FA_OK) return st;
  if (!workspace || !aligned16(workspace) || workspace_bytes < fa_forward_keymajor_workspace_size(B, H, N, d))
    return FA_ERR_WORKSPACE;
  fa::KeyMajorArgs a{};
  const int BH = B * H;
  if ((st = make_row_tile_map(&a.tm_q, q, BH, N, d)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_k, k, BH, N, d)) != FA_OK) return st;
  if ((st = make_row_tile_map(&a.tm_v, v, BH, N, d)) != FA_OK) return st;
  const size_t rows = static_cast<size_t>(BH) * N;
  char* ws = static_cast<char*>(workspace);
  a.ws_o = reinterpret_cast<float*>(ws);
  a.ws_m = reinterpret_cast<float*>(ws + round_up(rows * d * sizeof(float), 256));
  a.ws_r = reinterpret_cast<float*>(ws + round_up(rows * d * sizeof(float), 256) + round_up(rows * sizeof(float), 256));
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.scale_log2 = resolve_scale(scale, d) * kLog2e;
  a.causal = causal ? 1 : 0;
  a.o_f32 = (o_dtype == FA_F32) ? 1 : 0;
  return fa::launch_forward_keymajor(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_get_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned f = 0, b = 0, dcd = 0, km = 0, mg = 0;
  if (fa::read_clear_forward_status(&f, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_backward_status(&b, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_decode_status(&dcd, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_keymajor_status(&km, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_merge_status(&mg, s) != cudaSuccess) return FA_ERR_CUDA;
  const unsigned all = f | b | dcd | km | mg;
  if (all & 4u) return FA_ERR_BOUNDS;  // only the bounds-checked build sets it
  if (all & 1u) return FA_ERR_TIMEOUT;
  if (all != 0u) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o,
                          float* lse, fa_dtype o_dtype, long long rows, int d, void* stream) {
  if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  const uintptr_t l4 = reinterpret_cast<uintptr_t>(lse_a) | reinterpret_cast<uintptr_t>(lse_b) |
                       reinterpret_cast<uintptr_t>(lse);
  if ((l4 & 3u) != 0) return FA_ERR_INVALID_ARG;
  if (o_dtype != FA_BF16 && o_dtype != FA_F32) return FA_ERR_INVALID_ARG;
  if (rows < 0 || d < 4 || d % 4 != 0 || d > 4096) return FA_ERR_INVALID_ARG;
  if (rows == 0) return FA_OK;
  return fa::launch_merge(o_a, lse_a, o_b, lse_b, o, lse, rows, d, o_dtype == FA_F32 ? 1 : 0,
                          static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

int fa_decode_auto_split(int B, int H, int L) {
  if (B < 1 || H < 1 || L < 1) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    return 0;
  const long long bh = static_cast<long long>(B) * H;
  return fa::decode_auto_split(bh > 0x7FFFFFFFLL ? 0x7FFFFFFF : static_cast<int>(bh), L, sms);
}

fa_status fa_set_stats(unsigned long long* counters) {
  if ((reinterpret_cast<uintptr_t>(counters) & 7u) != 0) return FA_ERR_INVALID_ARG;
  t_stats = counters;
  return FA_OK;
}

fa_status fa_device_status(void* stream) { return fa_get_device_status(stream); }

fa_status fa_debug_abort_next_call(void) {
  t_abort_next = true;
  return FA_OK;
}

fa_status fa_debug_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 5000000000ull) return FA_ERR_INVALID_ARG;
  return fa::launch_wait_timeout_probe(limit_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                   : FA_ERR_CUDA;
}

}  // extern "C"
