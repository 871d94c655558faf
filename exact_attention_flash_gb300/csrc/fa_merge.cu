// Merge of two attention results over disjoint key sets, and the automatic split
// count of the decode path.
//
// What it computes ("attention_kernels.py", section 1 ``merge_states``): a softmax
// state (m, l, o) summarises a run of scores s with values v (m = max s,
// l = sum e^(s - m), o = sum e^(s - m) v), and two runs combine as
// m = max(m_a, m_b), l = l_a e^(m_a - m) + l_b e^(m_b - m), o likewise.  A
// normalised result (O = o / l, LSE = m + ln l) is the state (LSE, 1, O), so two
// results merge to  LSE = m + ln(w_a + w_b),  O = (w_a O_a + w_b O_b) / (w_a + w_b)
// with w = e^(LSE - m), m = max(LSE_a, LSE_b).  LSE = -inf is the empty run (the
// identity); two empty runs give O = 0 and LSE = -inf, as the page's guarded base
// (0 when both maxima are -inf) does.
//
// One warp per row, grid-stride over the rows; each lane moves 4 consecutive
// elements per access (16 bytes of fp32 or 8 of bf16), so a warp covers 128
// elements per instruction.  HBM-bound: 3 row reads / writes of O per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ unsigned g_merge_status;

struct Vec4 {
  float x[4];
};

__device__ __forceinline__ Vec4 load4(const void* base, long long idx, bool f32) {
  Vec4 r;
  if (f32) {
    const float4 t = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    r.x[0] = t.x, r.x[1] = t.y, r.x[2] = t.z, r.x[3] = t.w;
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + idx);
    r.x[0] = __uint_as_float(t.x << 16), r.x[1] = __uint_as_float(t.x & 0xFFFF0000u);
    r.x[2] = __uint_as_float(t.y << 16), r.x[3] = __uint_as_float(t.y & 0xFFFF0000u);
  }
  return r;
}

__device__ __forceinline__ void store4(void* base, long long idx, const Vec4& v, bool f32) {
  if (f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + idx) = make_float4(v.x[0], v.x[1], v.x[2], v.x[3]);
  } else {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x[0], v.x[1]), hi = __floats2bfloat162_rn(v.x[2], v.x[3]);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + idx) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
}

__global__ void __launch_bounds__(256) merge_kernel(const void* __restrict__ o_a, const float* __restrict__ lse_a,
                                                    const void* __restrict__ o_b, const float* __restrict__ lse_b,
                                                    void* o, float* lse, long long rows, int d, int f32) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const float la = lse_a[row], lb = lse_b[row];
    const float m = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f;
    if (m != -INFINITY) {  // both empty: O = 0, LSE = -inf
      wa = expf(la - m);
      wb = expf(lb - m);
    }
    const float s = wa + wb;
    const float inv = s > 0.f ? 1.f / s : 0.f;
    const float ca = wa * inv, cb = wb * inv;
    const long long base = row * d;
    for (int e = 4 * lane; e < d; e += 128) {
      if (!in_bounds(base + e + 3, rows * d, &g_merge_status)) continue;  // O rows [rows, d]
      const Vec4 va = load4(o_a, base + e, f32), vb = load4(o_b, base + e, f32);
      Vec4 r;
#pragma unroll
      for (int i = 0; i < 4; ++i) r.x[i] = ca * va.x[i] + cb * vb.x[i];
      store4(o, base + e, r, f32);
    }
    __syncwarp();  // every lane has read this row's LSE inputs before lane 0 may overwrite them in place
    if (lane == 0) lse[row] = m == -INFINITY ? -INFINITY : m + logf(s);
  }
}

}  // namespace

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o, float* lse,
                         long long rows, int d, int o_f32, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long blocks_needed = (rows + 7) / 8;  // 8 warps (rows at a time) per block
  const long long cap = static_cast<long long>(sms) * 16;
  const unsigned grid = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
  merge_kernel<<<grid, 256, 0, stream>>>(o_a, lse_a, o_b, lse_b, o, lse, rows, d, o_f32);
  return cudaGetLastError();
}

cudaError_t read_clear_merge_status(unsigned* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_merge_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_merge_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

int decode_auto_split(int BH, int L, int sms) {
  // Measured on GB300 (GB/s over n_split in 1..256 for B*H from 1 to 2048 and L from
  // 4 K to 128 K): throughput peaks with about four CTAs per SM in all, never fewer
  // than 8 splits, and segments of at least 512 keys.
  const long long by_sms = (4LL * sms + BH - 1) / BH;
  long long n = by_sms > 8 ? by_sms : 8;
  const long long max_by_len = L / 512 > 1 ? L / 512 : 1;
  if (n > max_by_len) n = max_by_len;
  return static_cast<int>(n < 1 ? 1 : n);
}

}  // namespace fa
