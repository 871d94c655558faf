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
// d = 64 and 128 (merge_kernel_t): every lane moves 16 bytes per access (4 fp32 or
// 8 bf16 elements), so a warp holds 1 to 4 whole rows, and each warp keeps two passes
// of rows in flight with all their loads issued before any result is used.  Other d
// (merge_kernel): one warp per row, 4 elements per lane and access.  Grid-stride over
// the rows; HBM-bound: 3 row reads / writes of O per row.
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

// d = 64 or 128: each lane moves 16 bytes per access (4 fp32 or 8 bf16 elements), so
// a row takes d / 4 or d / 8 lanes and a warp holds 1 to 4 rows; each warp keeps two
// passes of rows in flight, every load of both issued before any result is used.
template <int D, bool F32>
__global__ void __launch_bounds__(256) merge_kernel_t(const void* __restrict__ o_a, const float* __restrict__ lse_a,
                                                      const void* __restrict__ o_b, const float* __restrict__ lse_b,
                                                      void* o, float* lse, long long rows) {
  constexpr int kPerLane = F32 ? 4 : 8;
  constexpr int kLanesPerRow = D / kPerLane;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, col = kPerLane * (lane % kLanesPerRow);
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long gwarp = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (long long slot = gwarp; slot * kRowsPerPass < rows; slot += 2 * warps) {
    long long row[2];
    bool ok[2];
    float la[2], lb[2];
    uint4 ra[2], rb[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      row[u] = (slot + u * warps) * kRowsPerPass + sub;
      ok[u] = row[u] < rows && in_bounds(row[u] * D + col + kPerLane - 1, rows * D, &g_merge_status);
      if (ok[u]) {
        la[u] = lse_a[row[u]];
        lb[u] = lse_b[row[u]];
        const size_t off = static_cast<size_t>(row[u] * D + col) * (F32 ? 4 : 2);
        ra[u] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(o_a) + off);
        rb[u] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(o_b) + off);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!ok[u]) continue;
      const float m = fmaxf(la[u], lb[u]);
      float wa = 0.f, wb = 0.f;
      if (m != -INFINITY) {  // both empty: O = 0, LSE = -inf
        wa = expf(la[u] - m);
        wb = expf(lb[u] - m);
      }
      const float s = wa + wb;
      const float inv = s > 0.f ? 1.f / s : 0.f;
      const float ca = wa * inv, cb = wb * inv;
      const uint32_t a4[4] = {ra[u].x, ra[u].y, ra[u].z, ra[u].w}, b4[4] = {rb[u].x, rb[u].y, rb[u].z, rb[u].w};
      uint32_t r4[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (F32) {
          r4[w] = __float_as_uint(ca * __uint_as_float(a4[w]) + cb * __uint_as_float(b4[w]));
        } else {
          const float lo = ca * __uint_as_float(a4[w] << 16) + cb * __uint_as_float(b4[w] << 16);
          const float hi = ca * __uint_as_float(a4[w] & 0xFFFF0000u) + cb * __uint_as_float(b4[w] & 0xFFFF0000u);
          r4[w] = pack_bf16(lo, hi);
        }
      }
      const size_t off = static_cast<size_t>(row[u] * D + col) * (F32 ? 4 : 2);
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(o) + off) = make_uint4(r4[0], r4[1], r4[2], r4[3]);
      la[u] = m == -INFINITY ? -INFINITY : m + logf(s);
    }
    __syncwarp();  // every lane has read its rows' LSE inputs before they may be overwritten in place
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (ok[u] && col == 0) lse[row[u]] = la[u];
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
  const long long cap = static_cast<long long>(sms) * 16;
  if (d == 64 || d == 128) {
    const long long per_block = 8LL * 2 * (32 / (d / (o_f32 ? 4 : 8)));  // 8 warps, two passes of rows
    const long long blocks_needed = (rows + per_block - 1) / per_block;
    const unsigned grid = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
    if (d == 64 && o_f32) merge_kernel_t<64, true><<<grid, 256, 0, stream>>>(o_a, lse_a, o_b, lse_b, o, lse, rows);
    if (d == 64 && !o_f32) merge_kernel_t<64, false><<<grid, 256, 0, stream>>>(o_a, lse_a, o_b, lse_b, o, lse, rows);
    if (d == 128 && o_f32) merge_kernel_t<128, true><<<grid, 256, 0, stream>>>(o_a, lse_a, o_b, lse_b, o, lse, rows);
    if (d == 128 && !o_f32) merge_kernel_t<128, false><<<grid, 256, 0, stream>>>(o_a, lse_a, o_b, lse_b, o, lse, rows);
    return cudaGetLastError();
  }
  const long long blocks_needed = (rows + 7) / 8;  // 8 warps (rows at a time) per block
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
