// Forward in the first algorithm's loop order, for comparison with the main forward
// (fa_fwd.cu): key tiles outer, query tiles inner, and the running output, maximum
// and sum of every query row kept in device memory and repaired at every visit.
//
// What it computes ("flash_attention_numpy.py" ``flash_attention_tier1``; scale and
// causal skip / mask as in "attention_kernels.py" section 3): for key tile j and
// query tile i (128 x 128), s = Q_i K_j^T scale, m~ = rowmax s, p~ = exp(s - m~),
// r~ = rowsum p~; m' = max(m, m~), r' = e^(m - m') r + e^(m~ - m') r~ and
// O = (e^(m - m') r / r') O + e^(m~ - m') (p~ V_j) / r'.  At the end O is written in
// the output type and L = m + ln r.  Work is in base 2 (x = s log2 e).
//
// One CTA per (batch, head) walks its (j, i) pairs in that order, one at a time, as
// the first algorithm's GPU form parallelises over batch and heads only:
//   warp 4      TMA: K_j, V_j once per key tile, Q_i per pair
//   warp 5      MMA issuer: S = Q_i K_j^T (SS), then p~ V_j (TS, p~ from TMEM)
//   warps 0-3   thread = query row: p~ from S, then the repair of the row's O, m, r
//               in the fp32 workspace
// Nothing overlaps the steps of a pair; the point is the loop order, not speed.
// Tensor memory: S [0, 128), p~ V_j [128, 128 + d).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ unsigned g_fa1_status;

constexpr int kT = 128;  // rows of a query tile == keys of a key tile
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;

struct Fa1Shared {
  uint64_t kv_full, kv_empty, q_full, q_empty, s_full, p_full, pv_full, done, drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fa1_kernel(const __grid_constant__ KeyMajorArgs a) {
  constexpr int kTileBytes = kT * D * 2;
  constexpr int kChunks = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kTileBytes;
  __shared__ Fa1Shared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int n_t = (a.N + kT - 1) / kT;  // query tiles == key tiles
  auto first_i = [&](int j) { return a.causal ? j : 0; };  // query tiles that see key tile j

  if (tid == 0) {
    sh.abort = 0;
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.p_full, 4);  // one arrival per row warp
    mbar_init(&sh.pv_full, 1);
    mbar_init(&sh.done, 4);
    mbar_init(&sh.drain, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&sh.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0, jj = 0;
      bool ok = true;
      int kv_issued = 0, q_issued = 0;
      for (int j = 0; ok && j < n_t; ++j, ++jj) {
        if (jj > 0 && !mbar_wait(&sh.kv_empty, (jj - 1) & 1, &sh.abort, &g_fa1_status)) break;
        mbar_arrive_expect_tx(&sh.kv_full, 2 * kTileBytes);
        for (int c = 0; c < kChunks; ++c) {
          tma_load_3d(sK + c * (kT * 128), &a.tm_k, &sh.kv_full, c * 64, j * kT, bh);
          tma_load_3d(sV + c * (kT * 128), &a.tm_v, &sh.kv_full, c * 64, j * kT, bh);
        }
        ++kv_issued;
        for (int i = first_i(j); i < n_t; ++i, ++g) {
          if (g > 0 && !mbar_wait(&sh.q_empty, (g - 1) & 1, &sh.abort, &g_fa1_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.q_full, kTileBytes);
          for (int c = 0; c < kChunks; ++c)
            tma_load_3d(sQ + c * (kT * 128), &a.tm_q, &sh.q_full, c * 64, i * kT, bh);
          ++q_issued;
        }
      }
      // Every copy started must land before shared memory is released.
      if (kv_issued > 0) mbar_wait_drain(&sh.kv_full, (kv_issued - 1) & 1);
      if (q_issued > 0) mbar_wait_drain(&sh.q_full, (q_issued - 1) & 1);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one() ? 1u : 0u;
    constexpr uint32_t kIdS = idesc_bf16_f32(kT, kT, false, false);
    constexpr uint32_t kIdO = idesc_bf16_f32(kT, D, false, true);
    const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);        // K-major
    const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);        // K-major
    const uint64_t dV = sdesc_sw128(smem_u32(sV), kT * 128, 1024);  // MN-major
    int g = 0;
    bool ok = true;
    for (int j = 0, jj = 0; ok && j < n_t; ++j, ++jj) {
      if (!(ok = warp_wait(&sh.kv_full, jj & 1, &sh.abort, &g_fa1_status))) break;
      for (int i = first_i(j); i < n_t; ++i, ++g) {
        if (!(ok = warp_wait(&sh.q_full, g & 1, &sh.abort, &g_fa1_status))) break;
        // The row threads have read S and p~ V of the previous pair.
        if (g > 0 && !(ok = warp_wait(&sh.done, (g - 1) & 1, &sh.abort, &g_fa1_status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          umma_ss(tmem, desc_add(dQ, off), desc_add(dK, off), kIdS, kk > 0, leader);
        }
        umma_commit(&sh.s_full, leader);
        umma_commit(&sh.q_empty, leader);
        if (!(ok = warp_wait(&sh.p_full, g & 1, &sh.abort, &g_fa1_status))) break;
        tc_fence_after();
        // p~ V_j into a fresh accumulator: p~ is packed bf16 over S's first 64 columns.
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          umma_ts(tmem + kT, tmem + kk * 8, desc_add(dV, kk * 16 * 128), kIdO, kk > 0, leader);
        umma_commit(&sh.pv_full, leader);
      }
      if (ok) umma_commit(&sh.kv_empty, leader);
    }
    umma_commit(&sh.drain, leader);
    mbar_wait_drain(&sh.drain, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ rows (thread = query row of the tile)
    const int r = tid;  // TMEM lane
    const uint32_t s_tm = tmem_addr(tmem, (warp & 3) * 32, 0);
    const uint32_t pv_tm = tmem_addr(tmem, (warp & 3) * 32, kT);
    const float sl2 = a.scale_log2;
    int g = 0;
    bool ok = true;
    for (int j = 0; ok && j < n_t; ++j) {
      for (int i = first_i(j); i < n_t; ++i, ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sh.s_full, g & 1, &sh.abort, &g_fa1_status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int row = i * kT + r;
        const int key0 = j * kT;
        float x[kT];
        {
          uint32_t u[64];
          tmem_ld64(s_tm, u);
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(u[c]);
          tmem_ld64(s_tm + 64, u);
#pragma unroll
          for (int c = 0; c < 64; ++c) x[64 + c] = __uint_as_float(u[c]);
        }
        const int lim = a.causal ? min(a.N - 1, row) : a.N - 1;  // last visible key
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kT; ++c) {
          if (key0 + c > lim) x[c] = -INFINITY;
          mx = fmaxf(mx, x[c]);
        }
        const float mt = mx * sl2;                          // m~ (log2 units)
        const float nmt = mt == -INFINITY ? 0.f : -mt;      // a row with no visible key takes nothing
        float rt = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t u[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2(fmaf(x[64 * hf + 2 * c], sl2, nmt));
            const float p1 = ex2(fmaf(x[64 * hf + 2 * c + 1], sl2, nmt));
            rt += p0 + p1;
            u[c] = pack_bf16(p0, p1);
          }
          tmem_st32(s_tm + 32 * hf, u);
        }
        tc_fence_before();
        mbar_arrive_warp(&sh.p_full);
        if (!__all_sync(0xffffffffu, mbar_wait(&sh.pv_full, g & 1, &sh.abort, &g_fa1_status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t pv[D];
#pragma unroll
        for (int c = 0; c < D; c += 64) tmem_ld64(pv_tm + c, *reinterpret_cast<uint32_t (*)[64]>(pv + c));
        tc_fence_before();
        mbar_arrive_warp(&sh.done);  // S and p~ V may be overwritten by the next pair
        // the row's state in the [B*H, N] and [B*H, N, D] workspace arrays
        if (row < a.N && in_bounds(static_cast<long long>(bh) * a.N + row, static_cast<long long>(a.B) * a.H * a.N,
                                   &g_fa1_status)) {
          const size_t rix = static_cast<size_t>(bh) * a.N + row;
          float* orow = a.ws_o + rix * D;
          // The row's state before this visit (key tile 0 is every row's first visit).
          const float m_old = j == 0 ? -INFINITY : a.ws_m[rix];
          const float r_old = j == 0 ? 0.f : a.ws_r[rix];
          const float m_new = fmaxf(m_old, mt);
          const float base = m_new == -INFINITY ? 0.f : m_new;
          const float conv_old = m_old == -INFINITY ? 0.f : ex2(m_old - base);
          const float conv_new = mt == -INFINITY ? 0.f : ex2(mt - base);
          const float r_new = conv_old * r_old + conv_new * rt;
          const float inv = r_new > 0.f ? 1.f / r_new : 0.f;
          const float c_old = conv_old * r_old * inv, c_new = conv_new * inv;
#pragma unroll
          for (int c = 0; c < D; c += 4) {
            float4 o = j == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(orow + c);
            o.x = c_old * o.x + c_new * __uint_as_float(pv[c]);
            o.y = c_old * o.y + c_new * __uint_as_float(pv[c + 1]);
            o.z = c_old * o.z + c_new * __uint_as_float(pv[c + 2]);
            o.w = c_old * o.w + c_new * __uint_as_float(pv[c + 3]);
            *reinterpret_cast<float4*>(orow + c) = o;
          }
          a.ws_m[rix] = m_new;
          a.ws_r[rix] = r_new;
        }
      }
    }
    // Final pass: the output type and L = m + ln r, each thread for the rows it repaired.
    if (ok) {
      for (int i = 0; i < n_t; ++i) {
        const int row = i * kT + r;
        if (row >= a.N ||
            !in_bounds(static_cast<long long>(bh) * a.N + row, static_cast<long long>(a.B) * a.H * a.N, &g_fa1_status))
          continue;
        const size_t rix = static_cast<size_t>(bh) * a.N + row;
        const float* orow = a.ws_o + rix * D;
        for (int c = 0; c < D; c += 8) {
          const float4 u0 = *reinterpret_cast<const float4*>(orow + c);
          const float4 u1 = *reinterpret_cast<const float4*>(orow + c + 4);
          if (a.o_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.o) + rix * D + c);
            dst[0] = u0;
            dst[1] = u1;
          } else {
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + rix * D + c) =
                make_uint4(pack_bf16(u0.x, u0.y), pack_bf16(u0.z, u0.w), pack_bf16(u1.x, u1.y), pack_bf16(u1.z, u1.w));
          }
        }
        a.lse[rix] = (a.ws_m[rix] + __log2f(a.ws_r[rix])) * 0.6931471805599453f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int D>
cudaError_t launch_t(const KeyMajorArgs& a, cudaStream_t stream) {
  const int smem = 3 * kT * D * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(fa1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fa1_kernel<D><<<static_cast<unsigned>(a.B * a.H), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_keymajor(const KeyMajorArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_t<128>(a, stream);
  if (a.d == 64) return launch_t<64>(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_clear_keymajor_status(unsigned* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fa1_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_fa1_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
