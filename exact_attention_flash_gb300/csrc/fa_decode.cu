// Split-KV decoding ("Flash-Decoding") with the merge of the partial softmax
// states done inside the same kernel.
//
// Source: "attention_kernels.py" (CMU 15-779 lecture 5), section 5
// ``flash_decode`` — the keys of one (batch, head) are split into n_split
// segments at round(L * s / n_split), each segment is summarised by its softmax
// state (m, l, o) (section 1 ``SoftmaxState`` / ``state_of_scores``) and the
// states are folded left to right with ``merge_states``.  The page runs one
// thread block per segment and a small reduction kernel afterwards; here the
// last CTA of each (batch, head) to finish does the fold, in split order, so
// there is a single launch and the result is deterministic.
//
// The kernel is bound by HBM: every K and V byte is read exactly once.  Each
// group of d/8 lanes owns one key at a time and each lane holds 8 of the d
// components in a 16-byte vector; a CTA of 4 warps reads consecutive keys, so
// one load instruction of the CTA covers a contiguous run of keys, and each
// thread keeps 8 keys of K and V in flight before it uses them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include <mutex>

#include "fa_gb300.h"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ unsigned g_decode_status;

constexpr int kDecodeThreads = 128;
constexpr int kDecodeUnroll = 8;

// round(L * s / n) with ties to even, as Python's round() does on the exact value.
__device__ __forceinline__ int split_bound(long long L, int s, int n) {
  const long long num = L * static_cast<long long>(s);
  long long q = num / n;
  const long long r = num - q * n;
  if (2 * r > n || (2 * r == n && (q & 1))) q += 1;
  return static_cast<int>(q);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Merge state (m2, l2, o2) into (m, l, o); m in log2 units, the guarded base
// keeps two empty states (-inf, 0, 0) from producing NaN.
__device__ __forceinline__ void merge_into(float& m, float& l, float* o, float m2, float l2, const float* o2,
                                           int n) {
  const float mn = fmaxf(m, m2);
  const float base = (mn == -INFINITY) ? 0.f : mn;
  const float ca = ex2(m - base), cb = ex2(m2 - base);
  l = l * ca + l2 * cb;
  for (int i = 0; i < n; ++i) o[i] = o[i] * ca + o2[i] * cb;
  m = mn;
}

template <int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_split_kernel(DecodeArgs a) {
  constexpr int kLanesPerKey = D / 8;              // lanes sharing one key (8 components each)
  constexpr int kGroupsPerWarp = 32 / kLanesPerKey;
  constexpr int kGroups = kGroupsPerWarp * (kDecodeThreads / 32);
  constexpr int kStateStride = D + 2;

  __shared__ float sh_m[kGroups], sh_l[kGroups];
  __shared__ float sh_o[kGroups][D];
  __shared__ float sh_part[2];
  __shared__ int sh_last;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * a.H + h;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int sub = lane % kLanesPerKey;                     // which 8 components
  const int group = warp * kGroupsPerWarp + lane / kLanesPerKey;

  const int j0 = split_bound(a.L, split, a.n_split);
  const int j1 = split_bound(a.L, split + 1, a.n_split);

  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) + static_cast<size_t>(bh) * D;
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k) + static_cast<size_t>(bh) * a.L * D;
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v) + static_cast<size_t>(bh) * a.L * D;

  // Logical extents for the bounds-checked build: q and o [B*H, D], k and v
  // [B*H, L, D], the segment states [B*H, n_split, D + 2], the counters [B*H].
  const long long n_bh = static_cast<long long>(a.B) * a.H;
  float qf[8];
  bf16x8_to_float(in_bounds(static_cast<long long>(bh) * D + sub * 8 + 7, n_bh * D, &g_decode_status)
                      ? *reinterpret_cast<const uint4*>(qp + sub * 8)
                      : make_uint4(0u, 0u, 0u, 0u),
                  qf);
#pragma unroll
  for (int i = 0; i < 8; ++i) qf[i] *= a.scale_log2;

  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  // Every thread runs the same number of passes (the shuffles below involve
  // all 32 lanes); keys past the segment end are masked to -inf instead.
  for (int base0 = j0; base0 < j1; base0 += kGroups * kDecodeUnroll) {
    uint4 kr[kDecodeUnroll], vr[kDecodeUnroll];
#pragma unroll
    for (int u = 0; u < kDecodeUnroll; ++u) {
      const int key = base0 + u * kGroups + group;
      if (key < j1 && in_bounds((static_cast<long long>(bh) * a.L + key) * D + sub * 8 + 7, n_bh * a.L * D,
                                &g_decode_status)) {
        kr[u] = __ldcs(reinterpret_cast<const uint4*>(kp + static_cast<size_t>(key) * D + sub * 8));
        vr[u] = __ldcs(reinterpret_cast<const uint4*>(vp + static_cast<size_t>(key) * D + sub * 8));
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float s[kDecodeUnroll];
#pragma unroll
    for (int u = 0; u < kDecodeUnroll; ++u) {
      float kf[8];
      bf16x8_to_float(kr[u], kf);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
      for (int off = kLanesPerKey / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      s[u] = (base0 + u * kGroups + group < j1) ? dot : -INFINITY;
    }
    float mt = s[0];
#pragma unroll
    for (int u = 1; u < kDecodeUnroll; ++u) mt = fmaxf(mt, s[u]);
    const float m_new = fmaxf(m, mt);
    if (m_new != -INFINITY) {  // this group has seen at least one key
      const float alpha = ex2(m - m_new);
      l *= alpha;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= alpha;
#pragma unroll
      for (int u = 0; u < kDecodeUnroll; ++u) {
        const float p = ex2(s[u] - m_new);
        l += p;
        float vf[8];
        bf16x8_to_float(vr[u], vf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
      }
      m = m_new;
    }
  }

  // Fold the groups' states into the CTA's segment state.
  if (sub == 0) {
    sh_m[group] = m;
    sh_l[group] = l;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sh_o[group][sub * 8 + i] = acc[i];
  __syncthreads();

  float* ws = a.ws_partials + (static_cast<size_t>(bh) * a.n_split + split) * kStateStride;
  const long long n_states = n_bh * a.n_split;
  if (tid < D && in_bounds((static_cast<long long>(bh) * a.n_split + split + 1) * kStateStride - 1,
                           n_states * kStateStride, &g_decode_status)) {
    float pm = -INFINITY, pl = 0.f, po = 0.f;
    for (int g = 0; g < kGroups; ++g) merge_into(pm, pl, &po, sh_m[g], sh_l[g], &sh_o[g][tid], 1);
    ws[2 + tid] = po;
    if (tid == 0) {
      ws[0] = pm;
      ws[1] = pl;
      sh_part[0] = pm;
      sh_part[1] = pl;
    }
    if (a.partials != nullptr) {
      float* out = a.partials + (static_cast<size_t>(bh) * a.n_split + split) * kStateStride;
      out[2 + tid] = po;
      if (tid == 0) {
        out[0] = pm * 0.6931471805599453f;  // log2 units -> natural log
        out[1] = pl;
      }
    }
  }

  // The last CTA of this (batch, head) to arrive folds all segments in order.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    if (in_bounds(bh, n_bh, &g_decode_status)) {
      const unsigned prev = atomicAdd(&a.ws_counters[bh], 1u);
      sh_last = (prev == static_cast<unsigned>(a.n_split - 1)) ? 1 : 0;
    } else {
      sh_last = 0;
    }
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();

  if (tid < D && in_bounds((static_cast<long long>(bh) + 1) * a.n_split * kStateStride - 1, n_states * kStateStride,
                           &g_decode_status)) {
    const float* base = a.ws_partials + static_cast<size_t>(bh) * a.n_split * kStateStride;
    float fm = -INFINITY, fl = 0.f, fo = 0.f;
    for (int s = 0; s < a.n_split; ++s) {
      const float* st = base + static_cast<size_t>(s) * kStateStride;
      const float sm = __ldcg(st), sl = __ldcg(st + 1), so = __ldcg(st + 2 + tid);
      merge_into(fm, fl, &fo, sm, sl, &so, 1);
    }
    a.o[static_cast<size_t>(bh) * D + tid] = fo / fl;
    if (tid == 0) a.lse[bh] = (fm + __log2f(fl)) * 0.6931471805599453f;
  }
  if (tid == 0) a.ws_counters[bh] = 0u;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  dim3 grid(a.n_split, a.H, a.B);
  if (a.d == 128)
    decode_split_kernel<128><<<grid, kDecodeThreads, 0, stream>>>(a);
  else if (a.d == 64)
    decode_split_kernel<64><<<grid, kDecodeThreads, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t read_clear_decode_status(unsigned* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_decode_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_decode_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa

// ---------------------------------------------------------------------------
// Split-KV decode without caller-supplied scratch.
//
// fa_decode needs a workspace (segment states and arrival counters).  Some
// callers cannot provide one and may not call cudaMalloc either: a plugin or
// callback run by a host framework that owns all device memory and passes no
// workspace, or code on a latency-critical path where cudaMalloc's implicit
// device-wide synchronisation is not acceptable.  For them the library keeps
// one fixed scratch array in device memory, defined below.  It exists on every
// GPU that loads this library, for as long as the process lives.
//
// The array is shared by all calls: each call leaves its contents behind and
// the next call reuses them, so calls whose work overlaps on the GPU (other
// streams, other host threads) race on it and must be serialised by the caller.
namespace fa {
namespace {

static __device__ __align__(256) unsigned char g_decode_static_scratch[FA_DECODE_NOALLOC_SCRATCH_BYTES];

// Device address of the array, looked up once per device.  In host code the
// array's name is only a host-side stand-in, never a device address.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

cudaError_t static_scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_decode_noalloc(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                                       int H, int L, int d, float scale, int n_split, float* partials,
                                       void* stream) {
  // The same checks as fa_decode, with the fixed array as the workspace: a call
  // that needs more than FA_DECODE_NOALLOC_SCRATCH_BYTES returns FA_ERR_WORKSPACE
  // before any CUDA call.
  const fa_status st = fa::check_decode_args(q, k, v, o, lse, B, H, L, d, n_split,
                                             static_cast<size_t>(FA_DECODE_NOALLOC_SCRATCH_BYTES));
  if (st != FA_OK) return st;
  void* scratch = nullptr;
  if (fa::static_scratch_for_current_device(&scratch) != cudaSuccess) return FA_ERR_CUDA;
  // fa_decode clears the arrival counters it uses on `stream` (the previous call's
  // contents are still in the array) and launches on the array's address.
  return fa_decode(q, k, v, o, lse, B, H, L, d, scale, n_split, partials, scratch,
                   static_cast<size_t>(FA_DECODE_NOALLOC_SCRATCH_BYTES), stream);
}
