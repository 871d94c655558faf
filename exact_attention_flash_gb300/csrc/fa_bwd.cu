// Exact attention backward on sm_103a: P is recomputed from the stored
// log-sum-exp, nothing of size N x N is stored.
//
// What it computes ("attention_kernels.py", CMU 15-779 lecture 5, section 4
// ``flash_backward``; "lab.py" ``backward``): D = rowsum(dO * O); for each key
// tile j and query tile i, S = Q_i K_j^T * scale, P = exp(S - L_i),
// dV_j += P^T dO_i, dP = dO_i V_j^T, dS = P * (dP - D_i),
// dQ_i += dS K_j * scale, dK_j += dS^T Q_i * scale (the scale is folded into dS).
// Causal (query i at position q_start + i sees key j iff j <= q_start + i): query
// tiles that lie wholly before the key tile are skipped, the others are masked per
// element, and a key tile that no query sees gets zero dK and dV.
//
// Kernels:
//   bwd_preprocess  D/8 lanes per row: D = rowsum(dO * O), the per-query biases
//                   -LSE/scale and -D as tensor-core operand tiles, and dQ := 0.
//   bwd_kernel      one CTA per (128-key tile, batch*head); it walks the query
//                   tiles of 64 rows.  Keys are the TMEM lanes, so the kernel
//                   forms the transposed products:
//       S^T = K Q_i^T - LSE_i/scale and dP^T = V dO_i^T - D_i
//                                                (SS MMA, M=128, N=64; each
//                                                 accumulator starts from a
//                                                 K=16 bias product)
//       dV += P^T dO_i and dK += dS^T Q_i        (TS MMA, A = P^T / dS^T in TMEM)
//       dQ_i^T = K^T dS_i^T                      (SS MMA, M=d, N=64, dS from smem)
//   warp 16 loads (TMA), warp 17 issues MMAs, warp 18 waits on the mbarriers the
//   issuer depends on and hands each completion to it through a hardware named
//   barrier, warps 0-7 (thread = key, two warpgroups taking alternate steps) turn
//   S^T into P^T and then dP^T into dS^T, warps 8-15 (thread = feature) add dQ_i^T
//   into dQ with fp32 reductions in L2.  S^T/dP^T are double-buffered in TMEM so the
//   tensor core computes step n+1 while step n's elementwise work runs; dQ^T of step
//   n lands in the dP^T buffer (d = 128: after dK(n) has read dS^T(n) from it; d = 64:
//   dS^T(n) sits in the upper half of the S^T buffer, so dQ^T(n) goes before dK(n)).
// Tensor memory (512 columns): S^T[2] [0,64) [64,128), dP^T[2] [128,192)
// [192,256), dV [256, 256+d), dK [256+d, 256+2d).
// Gradients leave as fp32, or as bf16: the epilogue rounds dK and dV, and dQ is
// accumulated in an fp32 workspace buffer that dq_to_bf16 rounds after the grid.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ unsigned g_bwd_status;

constexpr int kBKV = 128;  // keys per CTA
constexpr int kBQ = 64;    // queries per step
// Warps 0-7: P^T / dS^T (two warpgroups, one per step parity) and warps 8-15: dQ
// writers (two warpgroups, one per half of the step's 64 query columns); warp 16:
// TMA producer; warp 17: MMA issuer; warp 18: the issuer's waits; warp 19 only
// lends its registers.
constexpr int kBwdThreads = 640;
constexpr int kWriterWarp0 = 8;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kWaitWarp = 18;
// Register split (setmaxnreg) by warpgroup: each P/dS thread holds a 64-query row of
// P in fp32 and 32 columns of dP^T, each dQ writer one 32-column row, the producer /
// MMA warps little.
// The sum stays within the CTA's launch allocation; the launcher checks it.
constexpr int kComputeRegs = 120;
constexpr int kWriterRegs = 72;
constexpr int kOtherRegs = 96;
constexpr int kRegsNeeded = 256 * kComputeRegs + 256 * kWriterRegs + 128 * kOtherRegs;
// dQ writer warps that read each step's dQ^T: all eight at d = 128; at d = 64 the four
// whose lane quarters hold that step's features (see the dQ writers).
template <int D>
constexpr int kDqWarpsPerStep = D == 64 ? 4 : 8;
// Where the P/dS warps wait for the dS tile of step n - 2 to have been read: at
// d = 128 just before they write step n's tile, so that the exponentials of step n
// never wait for dQ^T(n - 2), which the writers' pace holds back; at d = 64 at the
// top of the step, where the wait's own latency hides behind the wait for S^T.
template <int D>
constexpr bool kLateDsWait = D == 128;
// d = 64: dS^T is stored over columns [32, 64) of the S^T buffer (free once P^T sits
// packed in [0, 32) and S^T is in registers), which leaves the whole dP^T buffer free
// as soon as the P/dS warps have read dP^T, so dQ^T(n) is issued before dK(n) and the
// writers start earlier.  At d = 128, where the writers pace the step, issuing dQ^T
// first was slower (it delays dK(n) and the release of the step's Q/dO stage).
template <int D>
constexpr bool kDqBeforeDk = D == 64;

template <int D>
struct BwdCfg {
  static constexpr int kKVBytes = kBKV * D * 2;   // K or V tile
  static constexpr int kQBytes = kBQ * D * 2;     // Q or dO tile
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kDSBytes = kBKV * kBQ * 2; // dS tile (bf16), 16 KB
  static constexpr int kDVCol = 256;
  static constexpr int kDKCol = 256 + D;
  // Per step: the two bias tiles (B operands, 64 queries x 16, bf16): -LSE/scale
  // and -D, each split into three bf16 terms.  Their A operand is a constant
  // 128 x 16 tile with ones in columns 0-2.
  static constexpr int kBiasBytes = 2 * kBQ * 16 * 2;
  static constexpr int kOnesBytes = kBKV * 16 * 2;
  static constexpr int kSmemBytes =
      2 * kKVBytes + kStages * 2 * kQBytes + 2 * kDSBytes + kStages * kBiasBytes + kOnesBytes + 1024;
};

struct BwdShared {
  uint64_t kv_full;
  uint64_t q_full[4], q_empty[4];
  uint64_t s_full[2], dp_full[2], p_full[2], ds_full[2], dq_full[2], dq_empty[2], ds_empty[2];
  uint64_t dkdv_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk tensor store of a staged shared-memory box to global memory (rows past the
// tensor's extent are dropped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Named barrier over the 256 P/dS threads.
__device__ __forceinline__ void compute_bar_sync() { asm volatile("barrier.cta.sync 2, 256;" ::: "memory"); }

// Rendezvous of the MMA issuer and its waiting warp (named barrier 3, 64 threads),
// returning the AND of both warps' flags.  A wait on an mbarrier is a shared-memory
// access, which takes a few hundred cycles while the tensor core streams its
// operands from shared memory; the waiting warp absorbs that latency while the
// issuer is still queueing earlier products, and the hand-off itself is a hardware
// barrier.  Both warps take the same sequence of rendezvous and leave their loops
// on the same (shared) outcome, so neither can be left waiting.
__device__ __forceinline__ bool issuer_rendezvous(bool ok) { return bar_and(3, 64, ok); }

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const __grid_constant__ BackwardArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // K and V tiles.  At d = 64 V comes first: the A operand of dQ^T = K^T dS^T is K
  // in MN-major form, M = 128 rows of which d = 64 are features; with K right after
  // V, a descriptor that starts at V and puts its second 64-row chunk at K lands
  // dQ^T in TMEM lanes 64..127 (see the dQ writers).
  uint8_t* sV = smem + (D == 64 ? 0 : C::kKVBytes);
  uint8_t* sK = smem + (D == 64 ? C::kKVBytes : 0);
  uint8_t* sQ = smem + 2 * C::kKVBytes;                 // [kStages][kQBytes]
  uint8_t* sDO = sQ + C::kStages * C::kQBytes;          // [kStages][kQBytes]
  uint8_t* sDS = sDO + C::kStages * C::kQBytes;         // [2][kDSBytes]
  uint8_t* sBias = sDS + 2 * C::kDSBytes;               // [kStages][kBiasBytes]
  uint8_t* sOnes = sBias + C::kStages * C::kBiasBytes;  // [kOnesBytes]
  __shared__ BwdShared sh;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // Block order: heads in groups of a.head_group; within a group, the key tiles go
  // first to last across the group's heads (under causality key tile 0 meets the
  // most query tiles).  The longest blocks start first, which shortens the tail of
  // the grid, while only a group's Q, dO and dQ need to stay in L2.
  const int n_kv = (a.Nk + kBKV - 1) / kBKV;
  const int n_bh = a.B * a.H;
  const int hg = a.head_group;
  const int per_group = hg * n_kv;
  const int group = static_cast<int>(blockIdx.x) / per_group;
  const int g_heads = min(hg, n_bh - group * hg);  // the last group may be smaller
  const int g_idx = static_cast<int>(blockIdx.x) - group * per_group;
  const int bh = group * hg + g_idx % g_heads;
  const int j = g_idx / g_heads;
  const int key0 = j * kBKV;
  const int n_q = (a.Nq + kBQ - 1) / kBQ;
  // Under causality query i (at position q_start + i) sees key j iff j <= q_start + i,
  // so the first query block that sees any key of the tile holds query key0 - q_start.
  const int i_start = a.causal ? static_cast<int>(max(0LL, static_cast<long long>(key0) - a.q_start) / kBQ) : 0;
  const int n_steps = n_q - i_start;
  if (n_steps <= 0) {
    // No query sees these keys (they lie after the last query's position): their
    // gradients are zero.  Nothing else runs in this CTA.
    const int rows = min(kBKV, a.Nk - key0);
    const int row_bytes = D * (a.grad_bf16 ? 2 : 4);
    const size_t off = (static_cast<size_t>(bh) * a.Nk + key0) * row_bytes;
    uint4* dk4 = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.dk) + off);
    uint4* dv4 = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.dv) + off);
    // the tile's rows of dK and dV, in 16-byte pieces of [B, H, Nk, D]
    const long long pieces = static_cast<long long>(a.B) * a.H * a.Nk * row_bytes / 16;
    if (!in_bounds(static_cast<long long>(off / 16) + rows * row_bytes / 16 - 1, pieces, &g_bwd_status)) return;
    for (int i = tid; i < rows * row_bytes / 16; i += kBwdThreads) {
      dk4[i] = make_uint4(0u, 0u, 0u, 0u);
      dv4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }

  if (tid == 0) {
    sh.abort = 0;
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.q_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.dp_full[b], 1);
      mbar_init(&sh.p_full[b], 4);   // one arrival per P/dS warp of the step's warpgroup
      mbar_init(&sh.ds_full[b], 4);
      mbar_init(&sh.dq_full[b], 1);
      mbar_init(&sh.dq_empty[b], kDqWarpsPerStep<D>);  // one arrival per dQ writer warp of the step
      mbar_init(&sh.ds_empty[b], 1);
    }
    mbar_init(&sh.dkdv_full, 1);
    mbar_init(&sh.drain, 1);
    fence_barrier_init();
    // The key tile's K and V go out at once: their latency overlaps the rest of the
    // set-up (tensor-memory allocation, the ones tile).
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
    mbar_arrive_expect_tx(&sh.kv_full, 2 * C::kKVBytes);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(sK + c * (kBKV * 128), &a.tm_k, &sh.kv_full, c * 64, key0, bh);
      tma_load_3d(sV + c * (kBKV * 128), &a.tm_v, &sh.kv_full, c * 64, key0, bh);
    }
  }
  // The ones tile, in the no-swizzle K-major layout of 8-row x 16-byte core matrices:
  // even core matrices hold columns 0-7 (1, 1, 1, 0, ...), odd ones columns 8-15 (0).
  for (int i = tid; i < C::kOnesBytes / 16; i += kBwdThreads)
    reinterpret_cast<uint4*>(sOnes)[i] = ((i >> 3) & 1) ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  // Each role's code sits inside the branch that set its register budget.
  if (warp >= kProducerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kProducerWarp) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_do);
        // (K and V were issued during set-up.)  The bias tiles come from the preprocess kernel, which may still be running.
        griddep_wait();
        int issued = 0;
        for (int n = 0; n < n_steps; ++n) {
          const int s = n % C::kStages;
          if (n >= C::kStages && !mbar_wait(&sh.q_empty[s], ((n / C::kStages) - 1) & 1, &sh.abort, &g_bwd_status))
            break;
          const int q0 = (i_start + n) * kBQ;
          // The query block's bias tiles from the workspace (4 KB aligned): block blk of
          // the B * H * n_pad / 64 blocks.
          const size_t blk = static_cast<size_t>(bh) * (a.n_pad / kBQ) + (i_start + n);
          const bool bias_ok = in_bounds(static_cast<long long>(blk), static_cast<long long>(a.B) * a.H * (a.n_pad / kBQ),
                                         &g_bwd_status);
          mbar_arrive_expect_tx(&sh.q_full[s], 2 * C::kQBytes + (bias_ok ? C::kBiasBytes : 0));
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(sQ + s * C::kQBytes + c * (kBQ * 128), &a.tm_q, &sh.q_full[s], c * 64, q0, bh);
            tma_load_3d(sDO + s * C::kQBytes + c * (kBQ * 128), &a.tm_do, &sh.q_full[s], c * 64, q0, bh);
          }
          if (bias_ok) bulk_load(sBias + s * C::kBiasBytes, a.bias + blk * C::kBiasBytes, C::kBiasBytes, &sh.q_full[s]);
          ++issued;
        }
        mbar_wait_drain(&sh.kv_full, 0);
        for (int n = max(0, issued - C::kStages); n < issued; ++n)
          mbar_wait_drain(&sh.q_full[n % C::kStages], (n / C::kStages) & 1);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer
      {
        const uint32_t leader = elect_one() ? 1u : 0u;
        constexpr uint32_t kIdSdP = idesc_bf16_f32(kBKV, kBQ, false, false);  // S^T, dP^T
        constexpr uint32_t kIdKV = idesc_bf16_f32(kBKV, D, false, true);      // dV, dK (A in TMEM)
        constexpr uint32_t kIdQ = idesc_bf16_f32(128, kBQ, true, true);       // dQ^T = K^T dS^T
        // Descriptors are built once; each MMA only adds a constant offset (a short
        // issue path matters: the tensor core's queue is shallow).
        const uint64_t dK_k = sdesc_sw128(smem_u32(sK), 16, 1024);          // K, K-major (A of S^T)
        const uint64_t dV_k = sdesc_sw128(smem_u32(sV), 16, 1024);          // V, K-major (A of dP^T)
        const uint64_t dK_mn = sdesc_sw128(smem_u32(sK), kBKV * 128, 1024); // K as MN-major A of dQ^T
        // d = 64, odd steps: rows 0..63 read V (unused), rows 64..127 are K^T dS^T.
        const uint64_t dK_mn_hi = sdesc_sw128(smem_u32(sV), C::kKVBytes, 1024);
        const uint64_t dQ_k = sdesc_sw128(smem_u32(sQ), 16, 1024);          // Q stage 0, K-major (B of S^T)
        const uint64_t dDO_k = sdesc_sw128(smem_u32(sDO), 16, 1024);        // dO stage 0, K-major (B of dP^T)
        const uint64_t dQ_mn = sdesc_sw128(smem_u32(sQ), kBQ * 128, 1024);  // Q stage 0, MN-major (B of dK)
        const uint64_t dDO_mn = sdesc_sw128(smem_u32(sDO), kBQ * 128, 1024);// dO stage 0, MN-major (B of dV)
        const uint64_t dDS_mn = sdesc_sw128(smem_u32(sDS), kBKV * 128, 1024);// dS buffer 0, MN-major (B of dQ^T)
        const uint64_t dOnes = sdesc_k16_noswizzle(smem_u32(sOnes));        // A of the bias products
        const uint64_t dBias = sdesc_k16_noswizzle(smem_u32(sBias));        // bias tiles, stage 0
        // Per step n the products go in the order S^T(n+1), dV(n), dP^T(n+1), dK(n),
        // dQ^T(n) (d = 64: dQ^T(n) before dK(n)), each after a rendezvous with the
        // waiting warp (warp 18) that covers what it reads or overwrites:
        //   S^T(n+1)  Q(n+1) loaded; its buffer's previous user, dV(n-1), came earlier;
        //   dV(n)     P^T(n) in TMEM;
        //   dP^T(n+1) the dQ writers have read dQ^T(n-1) from the same buffer;
        //   dK(n), dQ^T(n)  dS^T(n) in TMEM and in shared memory.
        // Each accumulator of S^T / dP^T starts from its bias (one K = 16 product: ones
        // x the three bf16 terms), so it ends holding S^T - LSE/scale and dP^T - D.
        auto issue_s = [&](int n) {
          const int s = n % C::kStages;
          const uint64_t q_d = desc_add(dQ_k, s * C::kQBytes);
          const uint32_t s_tm = tmem + (n & 1) * kBQ;
          umma_ss(s_tm, dOnes, desc_add(dBias, s * C::kBiasBytes), kIdSdP, 0u, leader);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(s_tm, desc_add(dK_k, (kk >> 2) * (kBKV * 128) + (kk & 3) * 32),
                    desc_add(q_d, (kk >> 2) * (kBQ * 128) + (kk & 3) * 32), kIdSdP, 1u, leader);
          umma_commit(&sh.s_full[n & 1], leader);
        };
        auto issue_dp = [&](int n) {
          const int s = n % C::kStages;
          const uint64_t do_d = desc_add(dDO_k, s * C::kQBytes);
          const uint32_t dp_tm = tmem + 128 + (n & 1) * kBQ;
          umma_ss(dp_tm, dOnes, desc_add(dBias, s * C::kBiasBytes + C::kBiasBytes / 2), kIdSdP, 0u, leader);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(dp_tm, desc_add(dV_k, (kk >> 2) * (kBKV * 128) + (kk & 3) * 32),
                    desc_add(do_d, (kk >> 2) * (kBQ * 128) + (kk & 3) * 32), kIdSdP, 1u, leader);
          umma_commit(&sh.dp_full[n & 1], leader);
        };
        // P^T sits packed (queries 2c, 2c+1 in column c) in columns [0, 32) of the S^T
        // buffer, dS^T likewise in the dP^T buffer: K = 16 queries per 8 columns.
        auto pcol = [](int kk) { return kk * 8; };
        bool ok = issuer_rendezvous(true);  // K, V and Q(0) loaded
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        for (int n = 0; ok && n < n_steps; ++n) {
          const int s = n % C::kStages, b = n & 1;
          const bool next = n + 1 < n_steps;
          const uint32_t s_tm = tmem + b * kBQ;
          const uint32_t acc0 = n > 0 ? 1u : 0u;
          if (next) {
            if (!(ok = issuer_rendezvous(true))) break;
            tc_fence_after();
            issue_s(n + 1);
          }
          if (!(ok = issuer_rendezvous(true))) break;
          tc_fence_after();
          // dV += P^T dO_i   (K = 64 queries; dO_i is the MN-major B operand)
          const uint64_t do_d = desc_add(dDO_mn, s * C::kQBytes);
  #pragma unroll
          for (int kk = 0; kk < kBQ / 16; ++kk)
            umma_ts(tmem + C::kDVCol, s_tm + pcol(kk), desc_add(do_d, kk * 16 * 128), kIdKV, kk > 0 ? 1u : acc0, leader);
          if (next) {
            if (!(ok = issuer_rendezvous(true))) break;
            tc_fence_after();
            issue_dp(n + 1);
          }
          if (!(ok = issuer_rendezvous(true))) break;
          tc_fence_after();
          // dK += dS^T Q_i (dS^T packed in the dP^T buffer, or in the S^T buffer's upper
          // half when dQ^T goes first; see kDqBeforeDk).
          auto issue_dk = [&]() {
            const uint64_t q_d = desc_add(dQ_mn, s * C::kQBytes);
            const uint32_t ds_tm = kDqBeforeDk<D> ? s_tm + 32 : s_tm + 128;
  #pragma unroll
            for (int kk = 0; kk < kBQ / 16; ++kk)
              umma_ts(tmem + C::kDKCol, ds_tm + pcol(kk), desc_add(q_d, kk * 16 * 128), kIdKV, kk > 0 ? 1u : acc0, leader);
            umma_commit(&sh.q_empty[s], leader);
          };
          // dQ_i^T = K^T dS^T into the dP^T buffer, once nothing reads dS^T or dP^T there.
          // A = K as an MN-major [d x keys] operand.  For d = 64 only 64 of the M = 128
          // rows are features: even steps put them in lanes 0..63 (the other rows read
          // whatever follows K), odd steps in lanes 64..127 (the other rows read V), so
          // that the two halves of the dQ writers take alternate steps.
          auto issue_dq = [&]() {
            const uint64_t ds_d = desc_add(dDS_mn, b * C::kDSBytes);
            const uint64_t dq_a = (D == 64 && (n & 1)) ? dK_mn_hi : dK_mn;
  #pragma unroll
            for (int kk = 0; kk < kBKV / 16; ++kk)
              umma_ss(s_tm + 128, desc_add(dq_a, kk * 16 * 128), desc_add(ds_d, kk * 16 * 128), kIdQ, kk > 0, leader);
            umma_commit(&sh.dq_full[b], leader);
            umma_commit(&sh.ds_empty[b], leader);
          };
          if constexpr (kDqBeforeDk<D>) {
            issue_dq();
            issue_dk();
          } else {
            issue_dk();
            issue_dq();
          }
        }
        if (ok) umma_commit(&sh.dkdv_full, leader);
        umma_commit(&sh.drain, leader);
        mbar_wait_drain(&sh.drain, 0);
      }
      __syncwarp();
    } else if (warp == kWaitWarp) {
      // ------------------------------------------------------------ the issuer's waits
      // The same sequence of rendezvous as the MMA issuer, each after the wait that
      // the product issued next depends on.
      bool ok = warp_wait(&sh.kv_full, 0, &sh.abort, &g_bwd_status) &&
                warp_wait(&sh.q_full[0], 0, &sh.abort, &g_bwd_status);
      if (a.debug_abort) {  // failure-path test: act as if this wait had timed out
        if (lane == 0) raise_abort(&sh.abort, &g_bwd_status);
        ok = false;
      }
      ok = issuer_rendezvous(ok);
      for (int n = 0; ok && n < n_steps; ++n) {
        const int b = n & 1;
        const bool next = n + 1 < n_steps;
        if (next) {
          const int s1 = (n + 1) % C::kStages;
          if (!(ok = issuer_rendezvous(warp_wait(&sh.q_full[s1], ((n + 1) / C::kStages) & 1, &sh.abort, &g_bwd_status))))
            break;
        }
        if (!(ok = issuer_rendezvous(warp_wait(&sh.p_full[b], (n >> 1) & 1, &sh.abort, &g_bwd_status)))) break;
        if (next) {
          // dP^T(n+1) overwrites dQ^T(n-1)
          const bool w = n < 1 || warp_wait(&sh.dq_empty[(n - 1) & 1], ((n - 1) >> 1) & 1, &sh.abort, &g_bwd_status);
          if (!(ok = issuer_rendezvous(w))) break;
        }
        if (!(ok = issuer_rendezvous(warp_wait(&sh.ds_full[b], (n >> 1) & 1, &sh.abort, &g_bwd_status)))) break;
      }
    }
  } else if (warp < kWriterWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kComputeRegs));
    // ------------------------------------------------------------ P^T and dS^T (thread = key)
    // Warpgroup h takes the steps n with n % 2 == h, whose S^T, dP^T and dS buffers
    // are those of parity h, and forms P^T and then dS^T for all 64 queries of each.
    // So two steps are in flight: one warpgroup's exponentials of step n + 1 run
    // while the other still waits for dP^T(n) or forms dS^T(n), and P stays in
    // registers in fp32 from the exponentials to dS.
    const int k = tid & (kBKV - 1);
    const int h = warp >> 2;
    const int key = key0 + k;
    const int lane_base = (warp & 3) * 32;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int n = h; n < n_steps; n += 2) {
      const int b = n & 1;
      const int q0 = (i_start + n) * kBQ;
      // The dS tile of step n - 2 must have been read by dQ^T(n - 2) (see kLateDsWait).
      if ((!kLateDsWait<D> && n >= 2 &&
           !__all_sync(0xffffffffu, mbar_wait(&sh.ds_empty[b], ((n >> 1) - 1) & 1, &sh.abort, &g_bwd_status))) ||
          !__all_sync(0xffffffffu, mbar_wait(&sh.s_full[b], (n >> 1) & 1, &sh.abort, &g_bwd_status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = (a.causal && key0 + kBKV - 1 > a.q_start + q0) || (key0 + kBKV > a.Nk);
      const int first_visible_q = a.causal ? key - a.q_start : 0;  // queries before this one see nothing of the key
      const bool key_valid = key < a.Nk;
      const uint32_t s_tm = tmem_addr(tmem, lane_base, b * kBQ);
      const uint32_t dp_tm = tmem_addr(tmem, lane_base, 128 + b * kBQ);
      // S^T arrives holding S^T - LSE/scale (the bias came with the product).  The
      // exponentials are issued back to back (all arguments first, then all 64 ex2,
      // then the packs), so that the special-function unit's latency overlaps across
      // them instead of each result being waited for by its pack.
      float p[64];
      {
        uint32_t sv[64];
        tmem_ld64(s_tm, sv);
        const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float2 arg = __fmul2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2x2);
          p[e] = arg.x;
          p[e + 1] = arg.y;
        }
      }
#pragma unroll
      for (int e = 0; e < 64; ++e) p[e] = ex2(p[e]);
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (!key_valid || q0 + e < first_visible_q) p[e] = 0.f;
      }
      {
        // P^T packed (queries 2c, 2c+1 in column c) over columns [0, 32) of the
        // buffer, which this thread has already read.
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) pk[e / 2] = pack_bf16(p[e], p[e + 1]);
        tmem_st32(s_tm, pk);
      }
      tc_fence_before();
      mbar_arrive_warp(&sh.p_full[b]);
      if (!__all_sync(0xffffffffu, mbar_wait(&sh.dp_full[b], (n >> 1) & 1, &sh.abort, &g_bwd_status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dS^T = P^T * (dP^T - D); dP^T arrives holding dP^T - D.  The softmax scale of
      // dQ = dS K * scale and dK = dS^T Q * scale is applied here, once per element of
      // dS (rounding scale * dS to bf16 has the relative error of rounding dS), so the
      // dQ writers and the dK epilogue add and store the products as they are.  dP^T
      // is read 32 columns at a time, which keeps the fp32 P and dP^T within the
      // registers of this role.
      uint32_t dk[32];
      const float2 sc2 = make_float2(a.scale, a.scale);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dpv[32];
        tmem_ld32(dp_tm + 32 * half, dpv);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 ds2 = __fmul2_rn(__fmul2_rn(make_float2(p[32 * half + e], p[32 * half + e + 1]), sc2),
                                        make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])));
          dk[16 * half + e / 2] = pack_bf16(ds2.x, ds2.y);
        }
      }
      if (kLateDsWait<D> && n >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&sh.ds_empty[b], ((n >> 1) - 1) & 1, &sh.abort, &g_bwd_status))) {
        ok = false;
        break;
      }
      // dS^T row of this key into the MN-major, 128B-swizzled dS tile:
      // 16-byte piece j (queries 8j..8j+7) of row k sits at ((j ^ (k & 7)) * 16).
      uint8_t* ds_row = sDS + b * C::kDSBytes + (k >> 3) * 1024 + (k & 7) * 128;
#pragma unroll
      for (int piece = 0; piece < 8; ++piece)
        *reinterpret_cast<uint4*>(ds_row + ((piece ^ (k & 7)) << 4)) =
            make_uint4(dk[4 * piece], dk[4 * piece + 1], dk[4 * piece + 2], dk[4 * piece + 3]);
      tmem_st32(kDqBeforeDk<D> ? s_tm + 32 : dp_tm, dk);
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive_warp(&sh.ds_full[b]);
    }
    // ------------------------------------------------------------ dK, dV epilogue
    // Once the last products are done, the Q/dO/dS buffers are free: dK and dV are
    // staged there as boxes of 128 keys x 128 bytes (32 fp32 or 64 bf16 features)
    // with the 128-byte swizzle (16-byte piece j of row k at (j ^ (k % 8)) * 16, so
    // that the staging stores spread over all banks) and leave with bulk tensor
    // stores, one per box.  Warpgroup h handles features [h d/2, (h + 1) d/2).
    constexpr int kBoxBytes = kBKV * 128;  // 16 KB
    const int box_cols = a.grad_bf16 ? 64 : 32;  // features per box
    const int n_boxes = D / box_cols;            // per tensor
    const bool e_ok = ok && __all_sync(0xffffffffu, mbar_wait(&sh.dkdv_full, 0, &sh.abort, &g_bwd_status));
    if (e_ok) {
      tc_fence_after();
      uint8_t* stage_v = sQ;                        // boxes of dV, then of dK
      uint8_t* stage_k = sQ + n_boxes * kBoxBytes;
#pragma unroll 1
      for (int c = h * (D / 2); c < (h + 1) * (D / 2); c += 32) {
        uint32_t uv[32], uk[32];
        tmem_ld32(tmem_addr(tmem, lane_base, C::kDVCol + c), uv);
        tmem_ld32(tmem_addr(tmem, lane_base, C::kDKCol + c), uk);
        uint8_t* rv = stage_v + (c / box_cols) * kBoxBytes + k * 128;
        uint8_t* rk = stage_k + (c / box_cols) * kBoxBytes + k * 128;
        if (a.grad_bf16) {
          // 32 features = 64 bytes: pieces (c % 64) / 8 .. + 3 of the row
          const int j0 = (c % 64) / 8;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t* w = uv + 8 * j;
            const uint32_t* x = uk + 8 * j;
            *reinterpret_cast<uint4*>(rv + (((j0 + j) ^ (k & 7)) << 4)) =
                make_uint4(pack_bf16(__uint_as_float(w[0]), __uint_as_float(w[1])),
                           pack_bf16(__uint_as_float(w[2]), __uint_as_float(w[3])),
                           pack_bf16(__uint_as_float(w[4]), __uint_as_float(w[5])),
                           pack_bf16(__uint_as_float(w[6]), __uint_as_float(w[7])));
            *reinterpret_cast<uint4*>(rk + (((j0 + j) ^ (k & 7)) << 4)) =
                make_uint4(pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                           pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                           pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                           pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            *reinterpret_cast<uint4*>(rv + ((j ^ (k & 7)) << 4)) = make_uint4(uv[4 * j], uv[4 * j + 1], uv[4 * j + 2], uv[4 * j + 3]);
            *reinterpret_cast<uint4*>(rk + ((j ^ (k & 7)) << 4)) = make_uint4(uk[4 * j], uk[4 * j + 1], uk[4 * j + 2], uk[4 * j + 3]);
          }
        }
      }
      fence_proxy_async_smem();
    }
    compute_bar_sync();  // all boxes staged (or, after a failed wait, none)
    if (e_ok && tid == 0) {
      for (int i = 0; i < n_boxes; ++i) {
        tma_store_3d(&a.tm_dv, sQ + i * kBoxBytes, box_cols * i, key0, bh);
        tma_store_3d(&a.tm_dk, sQ + (n_boxes + i) * kBoxBytes, box_cols * i, key0, bh);
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      // The CTA may leave once the staged boxes have been read out of shared memory;
      // the global writes complete on their own (the grid's completion orders them
      // before any later work on the stream).
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kWriterRegs));
    // ------------------------------------------------------------ dQ writers (thread = feature)
    // dQ_i^T sits in TMEM with one feature per lane and one query per column.  Each
    // writer warpgroup takes 32 of the 64 query columns and adds them into dQ with
    // fp32 reductions in L2, straight from registers: for each query, a warp's 32
    // lanes cover 128 contiguous bytes of the dQ row.
    // d = 64: dQ^T of even steps is in lanes 0..63, of odd steps in lanes 64..127, so
    // the warps of lane quarters 0-1 reduce the even steps and those of quarters 2-3 the
    // odd ones: all eight warps work, each on every other step.
    const int half = (warp - kWriterWarp0) >> 2;  // query columns [32*half, 32*half + 32)
    const int lane_base = (warp & 3) * 32;        // this warp's TMEM lanes
    const int parity = D == 64 ? (warp & 3) >> 1 : -1;  // d = 64: the steps this warp takes
    const int feat0 = D == 64 ? lane_base & 32 : lane_base;  // feature of this warp's lane 0
    griddep_wait();  // dQ is zeroed by the preprocess kernel, which may still be running
    unsigned n_added = 0;  // dQ elements this thread added (fa_set_stats counters)
    for (int n = 0; n < n_steps; ++n) {
      const int b = n & 1;
      if (parity >= 0 && b != parity) continue;
      const int q0 = (i_start + n) * kBQ + 32 * half;
      if (!__all_sync(0xffffffffu, mbar_wait(&sh.dq_full[b], (n >> 1) & 1, &sh.abort, &g_bwd_status))) break;
      uint32_t v[32];
      tc_fence_after();
      tmem_ld32(tmem_addr(tmem, lane_base, 128 + b * kBQ + 32 * half), v);
      tc_fence_before();
      mbar_arrive_warp(&sh.dq_empty[b]);
      {
        // 4 x 4 transposes within each group of four lanes (two shuffle rounds per
        // block of four queries): lane 4g + i ends up with features 4g .. 4g + 3 of
        // queries 4k + i, which leave as 16-byte vector reductions.  One warp
        // instruction then covers four whole 128-byte row segments, a quarter of the
        // instructions of one reduction per feature.
        const int i4 = lane & 3;
        const long long dst_idx = (static_cast<long long>(bh) * a.Nq + q0 + i4) * D + feat0 + 4 * (lane >> 2);
        float* dst = a.dq + dst_idx;
        const int rows = min(32, a.Nq - q0);
        const long long dq_elems = static_cast<long long>(a.B) * a.H * a.Nq * D;
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) {
          const float x0 = __uint_as_float(v[4 * kq]), x1 = __uint_as_float(v[4 * kq + 1]);
          const float x2 = __uint_as_float(v[4 * kq + 2]), x3 = __uint_as_float(v[4 * kq + 3]);
          // Exchange 1 (lanes i, i ^ 1): even lanes keep queries 0 and 2, odd lanes 1 and 3,
          // each for both features of the pair.
          const bool odd = i4 & 1;
          const float r0 = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
          const float r1 = __shfl_xor_sync(0xffffffffu, odd ? x2 : x3, 1);
          const float a0 = odd ? r0 : x0, a1 = odd ? x1 : r0, a2 = odd ? r1 : x2, a3 = odd ? x3 : r1;
          // Exchange 2 (lanes i, i ^ 2): swap the other feature pair.
          const bool hi = i4 & 2;
          const float t0 = __shfl_xor_sync(0xffffffffu, hi ? a0 : a2, 2);
          const float t1 = __shfl_xor_sync(0xffffffffu, hi ? a1 : a3, 2);
          const float y0 = hi ? t0 : a0, y1 = hi ? t1 : a1, y2 = hi ? a2 : t0, y3 = hi ? a3 : t1;
          if (4 * kq + i4 < rows && in_bounds(dst_idx + 4LL * kq * D + 3, dq_elems, &g_bwd_status)) {
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + static_cast<size_t>(4 * kq) * D),
                         "f"(y0), "f"(y1), "f"(y2), "f"(y3)
                         : "memory");
            n_added += 4u;
          }
        }
      }
    }
    if (a.stats != nullptr) {  // one addition per warp and CTA
      const unsigned added = __reduce_add_sync(0xffffffffu, n_added);
      if (lane == 0 && added != 0u) atomicAdd(a.stats + 3, static_cast<unsigned long long>(added));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// b as three bf16 terms b1 + b2 + b3 (each the rounding of what the previous ones
// left), packed as the first three of eight bf16: about 24 significant bits.
__device__ __forceinline__ uint4 bias_terms(float b) {
  if (!isfinite(b)) return make_uint4(__bfloat16_as_ushort(__float2bfloat16_rn(b)), 0u, 0u, 0u);
  const __nv_bfloat16 b1 = __float2bfloat16_rn(b);
  const float r1 = b - __bfloat162float(b1);
  const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b2);
  const __nv_bfloat16 b3 = __float2bfloat16_rn(r2);
  return make_uint4(static_cast<uint32_t>(__bfloat16_as_ushort(b1)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b2)) << 16),
                    static_cast<uint32_t>(__bfloat16_as_ushort(b3)), 0u, 0u);
}

// D/8 lanes per row of the padded [B*H, n_pad] layout (several rows per warp),
// each lane owning 8 features in 16-byte accesses.  Rows q < N: D = rowsum(dO * O),
// the biases -LSE/scale and -D, and dQ := 0.  Padding rows q >= N: biases -inf and 0,
// so that a query past the end contributes P = 0.  The biases go into the query
// block's two bias tiles (64 rows x 16 bf16 each, no-swizzle K-major core matrices):
// row r's 32 bytes are two 16-byte pieces, columns 0-7 and 8-15.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess(const void* __restrict__ o, int o_f32,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse, uint8_t* __restrict__ bias,
                                                       float* __restrict__ dq, int N, int n_pad, long long padded_rows,
                                                       float inv_scale) {
  constexpr int kLanes = D / 8;                 // lanes per row
  constexpr int kRowsPerBlock = 256 / kLanes;
  griddep_launch_dependents();  // the backward kernel may start its own setup meanwhile
  const int sub = threadIdx.x % kLanes;         // 8-feature slice of the row
  const long long prow = static_cast<long long>(blockIdx.x) * kRowsPerBlock + threadIdx.x / kLanes;
  const bool live = prow < padded_rows;
  const long long bh = live ? prow / n_pad : 0;
  const int q = live ? static_cast<int>(prow - bh * n_pad) : 0;
  const long long n_bh = padded_rows / n_pad;  // B * H
  float acc = 0.f;
  if (live && q < N &&
      in_bounds((bh * N + q) * D + sub * 8 + 7, n_bh * N * D, &g_bwd_status)) {  // dO, O and dQ [B, H, N, D]
    const size_t base = static_cast<size_t>(bh * N + q) * D + sub * 8;
    const uint4 dv = *reinterpret_cast<const uint4*>(dout + base);
    float ov[8];
    if (o_f32) {
      const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base);
      const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base + 4);
      ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w; ov[4] = b.x; ov[5] = b.y; ov[6] = b.z; ov[7] = b.w;
    } else {
      const uint4 ob = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o) + base);
      const uint32_t w[4] = {ob.x, ob.y, ob.z, ob.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ov[2 * i] = __uint_as_float(w[i] << 16);
        ov[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(dw[i] << 16), ov[2 * i], acc);
      acc = fmaf(__uint_as_float(dw[i] & 0xFFFF0000u), ov[2 * i + 1], acc);
    }
    float4* z = reinterpret_cast<float4*>(dq + base);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // Sum over the row's lanes (aligned groups of kLanes within the warp).
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub < 4) {  // sub: tile (sub >> 1: 0 = LSE, 1 = D), piece (sub & 1)
    const bool lse_ok = q < N && in_bounds(bh * N + q, n_bh * N, &g_bwd_status);
    const float bs = lse_ok ? -lse[bh * N + q] * inv_scale : -INFINITY;
    const float bd = q < N ? -acc : 0.f;
    const int r = q & (kBQ - 1);
    const size_t tile_off = (static_cast<size_t>(bh) * (n_pad / kBQ) + q / kBQ) * (2 * kBQ * 32) + (sub >> 1) * (kBQ * 32);
    const int off = ((r >> 3) * 2 + (sub & 1)) * 128 + (r & 7) * 16;
    // 16-byte pieces of the B * H * n_pad * 64-byte workspace
    if (in_bounds(static_cast<long long>((tile_off + off) / 16), padded_rows * 4, &g_bwd_status))
      *reinterpret_cast<uint4*>(bias + tile_off + off) =
          (sub & 1) ? make_uint4(0u, 0u, 0u, 0u) : bias_terms((sub >> 1) ? bd : bs);
  }
}

// dQ for bf16 gradients: the fp32 accumulator rounded to bf16, 8 elements per thread
// and pass (two 16-byte loads, one 16-byte store).
__global__ void __launch_bounds__(256) dq_to_bf16(const float* __restrict__ src, uint4* __restrict__ dst, long long n8) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = s4[2 * i], b = s4[2 * i + 1];
    dst[i] = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
  }
}

template <int D>
cudaError_t launch_bwd_t(const BackwardArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const long long padded_rows = static_cast<long long>(a.B) * a.H * a.n_pad;
  constexpr int kRowsPerBlock = 256 / (D / 8);
  bwd_preprocess<D><<<static_cast<unsigned>((padded_rows + kRowsPerBlock - 1) / kRowsPerBlock), 256, 0, stream>>>(
      a.o, a.o_f32, static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.bias, a.dq, a.Nq, a.n_pad, padded_rows,
      1.f / a.scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split is granted from the CTA's launch allocation; refuse to
  // launch rather than let a raise wait for registers that do not exist.
  cudaFuncAttributes attr{};
  e = cudaFuncGetAttributes(&attr, bwd_kernel<D>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * kBwdThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  const long long ctas = static_cast<long long>(a.B) * a.H * ((a.Nk + kBKV - 1) / kBKV);
  if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  // A programmatic dependent of the preprocess kernel: its CTAs set up (barriers,
  // tensor memory, K and V) while the preprocess finishes, and wait for it only
  // where they read what it wrote.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, bwd_kernel<D>, a);
  if (e != cudaSuccess || !a.grad_bf16) return e;
  // bf16 gradients: dQ leaves its fp32 accumulator once every key tile has added to it.
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long n8 = static_cast<long long>(a.B) * a.H * a.Nq * (D / 8);
  const long long blocks = (n8 + 255) / 256, cap = 8LL * sms;
  dq_to_bf16<<<static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0, stream>>>(a.dq, static_cast<uint4*>(a.dq_out), n8);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_bwd_t<128>(a, stream);
  if (a.d == 64) return launch_bwd_t<64>(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_clear_backward_status(unsigned* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_bwd_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
