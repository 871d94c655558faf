// Exact attention forward on sm_103a: TMA tile loads, tcgen05 MMAs accumulating
// in tensor memory, online softmax in registers.
//
// What it computes ("attention_kernels.py", CMU 15-779 lecture 5, section 3
// ``flash_forward``; "lab.py" ``tiled``): for each query row, over key tiles,
// S = Q K^T * scale, m' = max(m, rowmax S), P = exp(S - m'), l = l * exp(m - m')
// + rowsum P, acc = acc * exp(m - m') + P V, and at the end O = acc / l and
// L = m + ln l.  Query row i sits at position q_start + i (0 for self-attention);
// causal: key j is visible to query i iff j <= q_start + i; key tiles wholly in
// the future of a query tile are skipped, and only tiles that straddle a row's
// last visible key are masked.
//
// GPU design (one CTA = two 128-row query tiles, 256 rows):
//   warp 8      TMA producer: claims work items (blocks of 256 query rows of one
//               head), loads both Q tiles of each, then its K and V tiles of 128
//               keys through a ring of shared-memory stages.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (SS MMA),
//               O_t += P_t V_j with P read from TMEM (TS MMA), interleaving the
//               two tiles so the tensor core works on one tile while the other
//               tile's softmax runs.  With d = 64 it issues the S products only,
//               and warps 10 and 11 issue tile 0's and tile 1's P V products.
//   warps 0-3   softmax for tile 0, warps 4-7 for tile 1: thread r owns query
//               row r (TMEM lane r), loads its row of S, takes the row max in
//               registers, writes P as bf16 over the S columns, and rescales its
//               row of O in TMEM when the running max grows by more than a factor 2^32
//               (the final O / l uses the same reference max, so this is exact).
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 and O_1 after.
// With d = 64 the last 128 columns hold P_0 and P_1 (64 each, bf16 pairs), so the
// issuer starts S_t of the next key tile as soon as the softmax has loaded S_t into
// registers; with d = 128, P overwrites the first half of S_t and the next S_t waits
// for the P V product that reads it.
// Work is done in base 2: x = S * scale * log2(e), p = 2^(x - m).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ unsigned g_fwd_status;

constexpr int kBM = 128;             // query rows per tile (TMEM lanes)
constexpr int kBN = 128;             // keys per KV tile
constexpr int kTiles = 2;            // query tiles per CTA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kFwdThreads = 384;  // warps 10-11: the P V issuers at d = 64; otherwise they only lend registers
// Register split (setmaxnreg): softmax warpgroups 0-1 raise their budget, warpgroup 2
// (producer, MMA issuer, two idle warps) lowers it.  The sum must stay within what
// the CTA was launched with; the launcher checks this against the compiled kernel.
constexpr int kSoftmaxRegs = 216;
constexpr int kOtherRegs = 72;
constexpr int kRegsNeeded = 256 * kSoftmaxRegs + 128 * kOtherRegs;
// Lazy rescaling: the reference max m of a row moves (and O is rescaled) only when
// a tile's max exceeds it by more than kRescaleThreshold log2 units, so the weights
// 2^(s - m) stay below 2^32.  fp32 and bf16 share one exponent range: the sum of N
// weights stays below 2^(32 + log2 N) and O below that times max|v|, inside fp32
// for N < 2^31 and |v| < 2^64.  When it moves, the reference is set kRescaleHeadroom
// units above the tile's max, so the row max may rise by threshold + headroom = 96
// units before the next rescale; the row's largest weight is then at least 2^-64,
// and weights that flush to zero (below 2^-126) are below 2^-62 of it, far under
// fp32's 2^-24.  The rescale factor 2^(m_old - m_new) flushes to zero when the max
// jumps by more than 126 - headroom units; the old terms it drops are then below
// 2^(threshold + headroom - 126) of the new largest weight, so threshold + headroom
// must stay at or below 102 (a headroom of 96 dropped terms as large as the new ones).
// Rounding of P to bf16 is relative, so neither constant changes the error of O;
// they only make rescales rare when the row max keeps rising (large logits), where
// the warp-wide rescale of O otherwise runs on most steps.
constexpr float kRescaleThreshold = 32.0f;
constexpr float kRescaleHeadroom = 64.0f;
static_assert(kRescaleThreshold + kRescaleHeadroom <= 102.0f, "a flushed rescale factor must drop only terms below 2^-24");
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;                // 128-byte swizzle chunks per row
  static constexpr int kTileBytes = kBM * D * 2;        // one 128-row bf16 tile
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kOCol = 256;                     // O_0 column; O_1 at kOCol + D
  // With d = 64 two tiles' S (2 x 128 columns) and O (2 x 64) leave 128 columns of
  // tensor memory free: P gets its own 64 columns per tile there, so the next S
  // product can overwrite S as soon as the softmax has loaded it (see kSPrefetch).
  static constexpr int kPCol = kOCol + kTiles * D;      // P_0 column; P_1 at kPCol + kBN / 2
  static_assert(D != 64 || kPCol + kTiles * kBN / 2 <= 512, "S, O and P fit the 512 columns at d = 64");
  static constexpr int kSmemBytes = kTiles * kTileBytes + kStages * 2 * kTileBytes + 1024;
};

// One work item: kTiles * kBM query rows of one (batch, head), and the number of
// key tiles each of its query tiles visits.
constexpr int kPvWarp0 = 10;  // with S prefetch, warps 10 and 11 issue tile 0's and tile 1's P V products
struct FwdItem {
  int bh, q_row0;
  int n_kv[kTiles];
};

constexpr int kItemRing = 2;
constexpr int kItemReaders = 1 + 2 * kBM / 32;  // arrivals per warp: the MMA warp and the softmax warps

struct FwdBarriers {
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  int item[kItemRing];
  FwdItem work[kItemRing];  // the item's fields, computed once by the producer
  uint64_t q_full[kTiles], q_empty[kTiles];
  uint64_t k_full[4], v_full[4], kv_empty[4], k_empty[4];  // k_empty: d = 128 (K released before V)
  uint64_t s_full[kTiles], p_half[kTiles], p_full[kTiles], o_full[kTiles], o_empty[kTiles];
  uint64_t s_free[kTiles], pv_done[kTiles];  // S-prefetch schedule only (d = 64)
  uint64_t drain, drain_pv[kTiles];
  uint32_t tmem_base;
  int abort;
};

// Work items in dispatch order: heads in groups of a.head_group; within a group, the
// query blocks go latest first across the group's heads (under causality the latest
// block has the most key tiles).  The longest items start first, which shortens the
// tail, while only a group's K and V need to stay in L2.
__device__ __forceinline__ FwdItem fwd_item(const ForwardArgs& a, int item) {
  const int n_qblk = (a.Nq + kBM * kTiles - 1) / (kBM * kTiles);
  const int n_bh = a.B * a.H;
  const int hg = a.head_group;
  const int per_group = hg * n_qblk;
  const int group = item / per_group;
  const int g_heads = min(hg, n_bh - group * hg);  // the last group may be smaller
  const int g_idx = item - group * per_group;
  FwdItem w;
  w.bh = group * hg + g_idx % g_heads;
  w.q_row0 = (n_qblk - 1 - g_idx / g_heads) * (kBM * kTiles);
  const int n_kv_total = (a.Nk + kBN - 1) / kBN;
  // Under causality the tile's last row, at position q_start + q_row0 + t kBM + kBM - 1,
  // sees the keys up to that position.
#pragma unroll
  for (int t = 0; t < kTiles; ++t)
    w.n_kv[t] = a.causal ? static_cast<int>(min(static_cast<long long>(n_kv_total),
                                                (static_cast<long long>(a.q_start) + w.q_row0 + t * kBM + kBM - 1) / kBN + 1))
                         : n_kv_total;
  return w;
}

template <int D, bool kPrecise>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ ForwardArgs a) {
  using C = FwdCfg<D>;
  // S prefetch (d = 64, standard precision): P_t lives in its own tensor-memory
  // columns, so S_t(j + 1) is issued as soon as the softmax has loaded S_t(j)
  // (s_free) instead of after P_t V(j) has read P from the S columns.  Each tile's
  // softmax then runs step after step without waiting for the tensor core; the
  // softmax waits for P_t V(j - 1) (pv_done) only before it overwrites P_t or
  // rescales O_t.  With d = 128 the columns are not there (S 2 x 128 + O 2 x 128).
  constexpr bool kSPrefetch = (D == 64) && !kPrecise;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // [kTiles][kTileBytes]
  uint8_t* sK = smem + kTiles * C::kTileBytes;          // [kStages][kTileBytes]
  uint8_t* sV = sK + C::kStages * C::kTileBytes;        // [kStages][kTileBytes]
  __shared__ FwdBarriers bars;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // Persistent: the producer claims items in dispatch order from a counter in the
  // caller's workspace (whichever CTA is free takes the next, longest first) and passes each index to
  // the MMA issuer and the softmax warps through a two-slot ring.  The barriers'
  // phases run on across items (one K/V ring, per-tile step counters, one Q and O
  // hand-off per item).
  const int n_items = a.B * a.H * ((a.Nq + kBM * kTiles - 1) / (kBM * kTiles));

  if (tid == 0) {
    bars.abort = 0;
    for (int r = 0; r < kItemRing; ++r) {
      mbar_init(&bars.item_full[r], 1);
      mbar_init(&bars.item_empty[r], kItemReaders + (kSPrefetch ? kTiles : 0));
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&bars.q_full[t], 1);
      mbar_init(&bars.q_empty[t], 1);
      mbar_init(&bars.o_empty[t], kBM / 32);  // one arrival per softmax warp of the tile
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.v_full[s], 1);
      // With S prefetch a stage is released by the issuer's S products and by each
      // tile's P V product (issued by that tile's softmax warps).
      mbar_init(&bars.kv_empty[s], kSPrefetch ? 1 + kTiles : 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_half[t], kBM / 32);  // one arrival per softmax warp of the tile
      mbar_init(&bars.p_full[t], kBM / 32);
      mbar_init(&bars.o_full[t], 1);
      mbar_init(&bars.s_free[t], kBM / 32);
      mbar_init(&bars.pv_done[t], 1);
    }
    for (int t = 0; t < kTiles; ++t) mbar_init(&bars.drain_pv[t], 1);
    mbar_init(&bars.drain, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&bars.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  // Each role's code sits inside the branch that set its register budget (the
  // compiler applies a budget to the code it dominates).
  if (warp >= kProducerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kProducerWarp) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
        int g = 0;                     // K/V tiles issued (the ring position)
        int q_issued[kTiles] = {0, 0};  // Q tiles issued per tile slot
        // fa_set_stats counters: S products of query tiles that start before N, and
        // the key tiles causality skipped for them (counted here, off the MMA issuer).
        unsigned n_tiles = 0, n_skipped = 0;
        const int n_kv_total = (a.Nk + kBN - 1) / kBN;
        bool ok = true;
        for (int it = 0; ok; ++it) {
          // Claim the next item and publish it (n_items once none is left).
          const int r = it % kItemRing;
          if (it >= kItemRing &&
              !mbar_wait(&bars.item_empty[r], ((it / kItemRing) - 1) & 1, &bars.abort, &g_fwd_status))
            break;
          const unsigned claimed = atomicAdd(a.sched, 1u);
          const int item = claimed < static_cast<unsigned>(n_items) ? static_cast<int>(claimed) : n_items;
          const FwdItem w = item < n_items ? fwd_item(a, item) : FwdItem{0, 0, {0, 0}};
          // The readers take the item's fields from the ring rather than computing them:
          // integer division by the run's sizes in an MMA issuer's code was measured to
          // slow every step of its issue loop.
          bars.item[r] = item;
          bars.work[r] = w;
          mbar_arrive(&bars.item_full[r]);
          if (item >= n_items) break;
#pragma unroll
          for (int t = 0; t < kTiles; ++t)
            if (w.q_row0 + t * kBM < a.Nq) {
              n_tiles += w.n_kv[t];
              n_skipped += n_kv_total - w.n_kv[t];
            }
          // Q tile t is reloaded once the previous item's last S_t product has read it.
          for (int t = 0; ok && t < kTiles; ++t) {
            if (it > 0 && !mbar_wait(&bars.q_empty[t], (it - 1) & 1, &bars.abort, &g_fwd_status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars.q_full[t], C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(sQ + t * C::kTileBytes + c * (kBM * 128), &a.tm_q, &bars.q_full[t], c * 64,
                          w.q_row0 + t * kBM, w.bh);
            ++q_issued[t];
          }
          for (int j = 0; ok && j < w.n_kv[kTiles - 1]; ++j) {
            const int s = g % C::kStages;
            // d = 128: K of a stage is released once both tiles' S products have read it,
            // V once both P V products have; K then loads about a step before V, so the
            // next S product does not wait for its K.
            if (g >= C::kStages &&
                !mbar_wait(kSPrefetch ? &bars.kv_empty[s] : &bars.k_empty[s], ((g / C::kStages) - 1) & 1, &bars.abort,
                           &g_fwd_status)) {
              ok = false;
              break;
            }
            uint8_t* k_dst = sK + s * C::kTileBytes;
            uint8_t* v_dst = sV + s * C::kTileBytes;
            // With S prefetch K and V of a key tile land on one barrier: the issuer then
            // tests one barrier per step (each test of an mbarrier costs it a few
            // hundred cycles while the tensor core streams operands from shared memory).
            uint64_t* v_bar = kSPrefetch ? &bars.k_full[s] : &bars.v_full[s];
            mbar_arrive_expect_tx(&bars.k_full[s], kSPrefetch ? 2 * C::kTileBytes : C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(k_dst + c * (kBN * 128), &a.tm_k, &bars.k_full[s], c * 64, j * kBN, w.bh);
            if (!kSPrefetch) {
              if (g >= C::kStages &&
                  !mbar_wait(&bars.kv_empty[s], ((g / C::kStages) - 1) & 1, &bars.abort, &g_fwd_status)) {
                mbar_wait_drain(&bars.k_full[s], (g / C::kStages) & 1);  // the K copy just issued lands first
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(v_bar, C::kTileBytes);
            }
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(v_dst + c * (kBN * 128), &a.tm_v, v_bar, c * 64, j * kBN, w.bh);
            ++g;
          }
        }
        // Drain: every copy this CTA started must land before shared memory is released.
        for (int t = 0; t < kTiles; ++t)
          if (q_issued[t] > 0) mbar_wait_drain(&bars.q_full[t], (q_issued[t] - 1) & 1);
        for (int gg = max(0, g - C::kStages); gg < g; ++gg) {
          const int s = gg % C::kStages;
          mbar_wait_drain(&bars.k_full[s], (gg / C::kStages) & 1);
          if (!kSPrefetch) mbar_wait_drain(&bars.v_full[s], (gg / C::kStages) & 1);
        }
        if (a.stats != nullptr) {
          if (n_tiles != 0u) atomicAdd(a.stats + 0, static_cast<unsigned long long>(n_tiles));
          if (n_skipped != 0u) atomicAdd(a.stats + 1, static_cast<unsigned long long>(n_skipped));
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer
      {
        const uint32_t leader = elect_one() ? 1u : 0u;
        constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false, false);
        constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D, false, true);
        // Descriptors are built once; each MMA only adds a constant offset, which keeps
        // the single issuing thread's path short (the tensor core's queue is shallow).
        const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);         // Q tile 0, K-major
        const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);         // K stage 0, K-major
        const uint64_t dV = sdesc_sw128(smem_u32(sV), kBN * 128, 1024);  // V stage 0, MN-major
        auto issue_s = [&](int t, int s) {  // S_t from the K tile in ring stage s
          const uint64_t q_d = desc_add(dQ, t * C::kTileBytes), k_d = desc_add(dK, s * C::kTileBytes);
          const uint32_t s_tm = tmem + t * kBN;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
            umma_ss(s_tm, desc_add(q_d, off), desc_add(k_d, off), kIdS, kk > 0, leader);
          }
          umma_commit(&bars.s_full[t], leader);
        };
        // O_t += P_t V_j in two halves of 64 keys: the softmax releases P's first
        // half (p_half) while it still computes the second (p_full).  s: ring stage of
        // V_j; step: the tile's step count across items (the P barriers' phase);
        // first: the item's first key tile (O is written, not accumulated).
        auto issue_pv = [&](int t, int s, int step, bool first) -> bool {
          const uint64_t v_d = desc_add(dV, s * C::kTileBytes);
          const uint32_t o_tm = tmem + C::kOCol + t * D;
          const uint32_t p_tm = kSPrefetch ? tmem + C::kPCol + t * (kBN / 2) : tmem + t * kBN;
          const uint32_t acc0 = first ? 0u : 1u;
          if (!kSPrefetch) {
            if (!warp_wait(&bars.p_half[t], step & 1, &bars.abort, &g_fwd_status)) return false;
            tc_fence_after();
          } else {  // with S prefetch the next S_t does not wait for this product: one hand-off
            if (!warp_wait(&bars.p_full[t], step & 1, &bars.abort, &g_fwd_status)) return false;
            tc_fence_after();
          }
  #pragma unroll
          for (int kk = 0; kk < kBN / 32; ++kk)
            umma_ts(o_tm, p_tm + kk * 8, desc_add(v_d, kk * 16 * 128), kIdO, kk > 0 ? 1u : acc0, leader);
          if (!kSPrefetch) {
            if (!warp_wait(&bars.p_full[t], step & 1, &bars.abort, &g_fwd_status)) return false;
            tc_fence_after();
          }
  #pragma unroll
          for (int kk = kBN / 32; kk < kBN / 16; ++kk)
            umma_ts(o_tm, p_tm + kk * 8, desc_add(v_d, kk * 16 * 128), kIdO, 1u, leader);
          if (kPrecise) {
  #pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ts(o_tm, p_tm + 64 + kk * 8, desc_add(v_d, kk * 16 * 128), kIdO, 1u, leader);
          }
          return true;
        };
        int g = 0;                  // K/V tiles consumed (the ring position)
        int step[kTiles] = {0, 0};  // per-tile steps before the current item
        bool ok = true;
        for (int it = 0; ok; ++it) {
          const int r = it % kItemRing;
          if (!warp_wait(&bars.item_full[r], (it / kItemRing) & 1, &bars.abort, &g_fwd_status)) break;
          const int item = bars.item[r];
          const FwdItem w = bars.work[r];
          mbar_arrive_warp(&bars.item_empty[r]);
          if (item >= n_items) break;
          const int s0 = g % C::kStages;
          ok = warp_wait(&bars.k_full[s0], (g / C::kStages) & 1, &bars.abort, &g_fwd_status);
          if constexpr (kSPrefetch) {
            // S products only: each tile's softmax warps issue their own P V products.
            // Stage s of the K/V ring is released once the S products that read K and
            // both tiles' P V products that read V have completed; this thread arrives
            // once for its S products and once more for each tile that has no P V with
            // that key tile (tile 0 may need one key tile fewer).
            const auto release_kv = [&](int jj, int stage) {
              umma_commit(&bars.kv_empty[stage], leader);
              for (int t = 0; t < kTiles; ++t)
                if (jj >= w.n_kv[t]) umma_commit(&bars.kv_empty[stage], leader);
            };
            // The item's first S_t: Q_t reloaded, and S_t of the previous item's last
            // step loaded by the softmax.
            for (int t = 0; ok && t < kTiles; ++t) {
              if (!warp_wait(&bars.q_full[t], it & 1, &bars.abort, &g_fwd_status) ||
                  (step[t] > 0 &&
                   !warp_wait(&bars.s_free[t], (step[t] - 1) & 1, &bars.abort, &g_fwd_status))) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(t, s0);
              if (w.n_kv[t] == 1) umma_commit(&bars.q_empty[t], leader);  // its only S_t has read Q_t
            }
            if (ok) release_kv(0, s0);
            for (int j = 0; ok && j + 1 < w.n_kv[kTiles - 1]; ++j, ++g) {
              const int sn = (g + 1) % C::kStages;
              const uint32_t phn = ((g + 1) / C::kStages) & 1;
              // S_t(j + 1) once the softmax has loaded S_t(j) and K(j + 1) has landed.
              if (!warp_wait(&bars.k_full[sn], phn, &bars.abort, &g_fwd_status)) {
                ok = false;
                break;
              }
              for (int t = 0; t < kTiles; ++t) {
                if (j + 1 >= w.n_kv[t]) continue;
                if (!warp_wait(&bars.s_free[t], (step[t] + j) & 1, &bars.abort, &g_fwd_status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_s(t, sn);
                if (j + 2 == w.n_kv[t]) umma_commit(&bars.q_empty[t], leader);  // the item's last S_t
              }
              if (ok) release_kv(j + 1, sn);
            }
            ++g;  // the item's last key tile
          } else {
            for (int t = 0; ok && t < kTiles; ++t) {
              if (!warp_wait(&bars.q_full[t], it & 1, &bars.abort, &g_fwd_status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(t, s0);
              if (t == kTiles - 1) umma_commit(&bars.k_empty[s0], leader);  // both S products have read K
            }
            for (int j = 0; ok && j < w.n_kv[kTiles - 1]; ++j, ++g) {
              const int s = g % C::kStages, sn = (g + 1) % C::kStages;
              const uint32_t phn = ((g + 1) / C::kStages) & 1;
              if (!warp_wait(&bars.v_full[s], (g / C::kStages) & 1, &bars.abort, &g_fwd_status)) {
                ok = false;
                break;
              }
              bool k_next = false;  // K(j + 1) tested once per step (for the first tile that needs it)
              for (int t = 0; t < kTiles; ++t) {
                if (j >= w.n_kv[t]) continue;  // tile 0 may need one key tile fewer
                // The item's first P V_t overwrites O_t: the previous item's epilogue must
                // have read O_t out of tensor memory.
                if (j == 0 && it > 0 && !warp_wait(&bars.o_empty[t], (it - 1) & 1, &bars.abort, &g_fwd_status)) {
                  ok = false;
                  break;
                }
                if (!issue_pv(t, s, step[t] + j, j == 0)) {
                  ok = false;
                  break;
                }
                if (t == kTiles - 1) umma_commit(&bars.kv_empty[s], leader);
                if (j + 1 < w.n_kv[t]) {
                  if (!k_next && !warp_wait(&bars.k_full[sn], phn, &bars.abort, &g_fwd_status)) {
                    ok = false;
                    break;
                  }
                  k_next = true;
                  tc_fence_after();
                  issue_s(t, sn);
                  if (t == kTiles - 1) umma_commit(&bars.k_empty[sn], leader);  // both S products have read K
                } else {
                  umma_commit(&bars.o_full[t], leader);   // O_t of this item is complete
                  umma_commit(&bars.q_empty[t], leader);  // its last S_t product has read Q_t
                }
              }
            }
          }
          for (int t = 0; t < kTiles; ++t) step[t] += w.n_kv[t];
        }
        // Drain: all MMAs complete before tensor memory is released.
        umma_commit(&bars.drain, leader);
        mbar_wait_drain(&bars.drain, 0);
      }
      __syncwarp();
    } else if (kSPrefetch && warp < kPvWarp0 + kTiles) {
      // ------------------------------------------------------------ P V issuer of tile t
      // Walks the same items and steps as the tile's softmax warps: O_t += P_t V(j)
      // once the four warps have written P_t(j) (p_full).  Each mbarrier test costs a
      // few hundred cycles while the tensor core streams operands from shared memory,
      // and the tensor core's queue is shallow, so issuing eight MMAs can stall the
      // issuing thread for several hundred more: with a warp of its own per tile,
      // neither falls on the S products' issuer nor on the softmax.  The item's first
      // product overwrites O_t; the softmax warps read O_t out in the previous item's
      // epilogue, before they hand over that item's first P_t.
      const int t = warp - kPvWarp0;
      const uint32_t leader = elect_one() ? 1u : 0u;
      const uint64_t dV = sdesc_sw128(smem_u32(sV), kBN * 128, 1024);  // V stage 0, MN-major
      const uint32_t o_mma = tmem + C::kOCol + t * D, p_mma = tmem + C::kPCol + t * (kBN / 2);
      constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D, false, true);
      int kv_pos = 0;  // K/V tiles of the items before this one (the ring position)
      int step = 0;    // the tile's steps across items (the P barriers' phase)
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int ring = it % kItemRing;
        if (!warp_wait(&bars.item_full[ring], (it / kItemRing) & 1, &bars.abort, &g_fwd_status)) break;
        const int item = bars.item[ring];
        const FwdItem w = bars.work[ring];
        mbar_arrive_warp(&bars.item_empty[ring]);
        if (item >= n_items) break;
        const int n_kv_t = t == 0 ? w.n_kv[0] : w.n_kv[1];
        for (int j = 0; j < n_kv_t; ++j, ++step) {
          if (!warp_wait(&bars.p_full[t], step & 1, &bars.abort, &g_fwd_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int stage = (kv_pos + j) % C::kStages;
          const uint64_t v_d = desc_add(dV, stage * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_ts(o_mma, p_mma + kk * 8, desc_add(v_d, kk * 16 * 128), kIdO, (j > 0 || kk > 0) ? 1u : 0u, leader);
          umma_commit(&bars.pv_done[t], leader);
          umma_commit(&bars.kv_empty[stage], leader);
        }
        kv_pos += w.n_kv[kTiles - 1];
      }
      // Every P V product issued here completes before tensor memory is released.
      umma_commit(&bars.drain_pv[t], leader);
      if (lane == 0) mbar_wait_drain(&bars.drain_pv[t], 0);
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                  // query tile of this warpgroup
    const int r = tid - t * kBM;              // row within the tile == TMEM lane
    const int lane_base = (warp & 3) * 32;    // TMEM lane quarter of this warp
    const uint32_t s_tm = tmem_addr(tmem, lane_base, t * kBN);
    const uint32_t o_tm = tmem_addr(tmem, lane_base, C::kOCol + t * D);
    // P_t: over the first 64 columns of S_t, or in its own columns with S prefetch.
    const uint32_t p_tm = kSPrefetch ? tmem_addr(tmem, lane_base, C::kPCol + t * (kBN / 2)) : s_tm;
    const float sl2 = a.scale_log2;
    int step = 0;  // this tile's steps across items (the S and P barriers' phase)
    unsigned n_rescales = 0;  // running-max growths of this row (fa_set_stats counters)
    bool ok = true;
    if (a.debug_abort) {  // failure-path test: act as if the first wait had timed out
      if (lane == 0) raise_abort(&bars.abort, &g_fwd_status);
      ok = false;  // nothing is handed over, so the other roles' next waits give up too
    }
    for (int it = 0; ok; ++it) {
    const int ring = it % kItemRing;
    if (!__all_sync(0xffffffffu, mbar_wait(&bars.item_full[ring], (it / kItemRing) & 1, &bars.abort, &g_fwd_status)))
      break;
    const int item = bars.item[ring];
    const FwdItem w = bars.work[ring];
    mbar_arrive_warp(&bars.item_empty[ring]);
    if (item >= n_items) break;
    const int q_row0 = w.q_row0, bh = w.bh;
    const int row = q_row0 + t * kBM + r;
    float mx_seen = -INFINITY;  // true running max of the raw scores (counters only)
    float m_run = -INFINITY;  // reference max (scaled, log2 units)
    float l_run = 0.f;  // sum of p: the log-sum-exp
    float l_hat = 0.f;  // sum of the bf16-rounded p that enter P V: the normaliser of O
    for (int j = 0; j < w.n_kv[t]; ++j, ++step) {
      // Lanes leave together: the TMEM accesses below are warp-collective.
      if (!__all_sync(0xffffffffu, mbar_wait(&bars.s_full[t], step & 1, &bars.abort, &g_fwd_status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kBN];
      {
        uint32_t u[64];
        tmem_ld64(s_tm, u);
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(u[i]);
        tmem_ld64(s_tm + 64, u);
#pragma unroll
        for (int i = 0; i < 64; ++i) x[64 + i] = __uint_as_float(u[i]);
      }
      if constexpr (kSPrefetch) {  // S_t is in registers: the next S_t product may overwrite it
        tc_fence_before();
        mbar_arrive_warp(&bars.s_free[t]);
      }
      const int key0 = j * kBN;
      const bool need_mask = (key0 + kBN > a.Nk) || (a.causal && key0 + kBN - 1 > a.q_start + q_row0 + t * kBM);
      if (need_mask) {
        const int lim = a.causal ? min(a.Nk - 1, a.q_start + row) : a.Nk - 1;  // last visible key
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (key0 + i > lim) x[i] = -INFINITY;
      }
      // Row max as eight independent chains of 3-input maxima (short dependency paths).
      float mx8[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float v = fmax3(x[16 * c], x[16 * c + 1], x[16 * c + 2]);
#pragma unroll
        for (int i = 3; i < 15; i += 2) v = fmax3(v, x[16 * c + i], x[16 * c + i + 1]);
        mx8[c] = fmaxf(v, x[16 * c + 15]);
      }
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      if (a.stats != nullptr) {  // counters only (a uniform branch on a kernel argument)
        n_rescales += (row < a.Nq && mx > mx_seen && mx_seen != -INFINITY) ? 1u : 0u;
        mx_seen = fmaxf(mx_seen, mx);
      }
      const float m_tile = mx * sl2;
      float m_use = m_run;
      float alpha = 1.f;
      if (m_tile > m_run + kRescaleThreshold) {
        m_use = m_tile + kRescaleHeadroom;
        alpha = ex2(m_run - m_use);  // 0 on the first tile
      }
      // Rescale this row of O when the reference max moved (not on the first
      // tile: O is written, not accumulated, by the first PV).  With S prefetch
      // this waits for the previous P V product (below, before P_t is written).
      const auto rescale_o = [&]() {
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // 32 columns at a time (a wider load spills next to the row of S held in
          // registers); the stores are waited for once, at the end.
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t u[32];
            tmem_ld32(o_tm + c, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
            tmem_st32_nowait(o_tm + c, u);
          }
          tmem_wait_st();
        }
      };
      if constexpr (!kSPrefetch) rescale_o();
      const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use;
      const float2 sl2x2 = make_float2(sl2, sl2), negm2 = make_float2(neg_m, neg_m);
      float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // P of keys [64 half, 64 half + 64): the arguments, then all 64 exponentials back to
      // back (so that the special-function unit's latency overlaps across them instead of
      // each result being waited for by its pack), then the packs and sums.  x keeps p,
      // or with precise its bf16 rounding residual for the second P V product.
      const auto exp_half = [&](int half, uint32_t (&u)[32]) {
        float* xh = x + half * 64;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 e = __ffma2_rn(make_float2(xh[2 * i], xh[2 * i + 1]), sl2x2, negm2);
          xh[2 * i] = e.x;
          xh[2 * i + 1] = e.y;
        }
#pragma unroll
        for (int k = 0; k < 64; ++k) xh[k] = ex2(xh[k]);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = xh[2 * i], p1 = xh[2 * i + 1];
          u[i] = pack_bf16(p0, p1);
          sum2[i & 3] = __fadd2_rn(sum2[i & 3], make_float2(p0, p1));
          if (kPrecise) {  // keep the rounding residual for the second PV product
            xh[2 * i] = p0 - __uint_as_float(u[i] << 16);
            xh[2 * i + 1] = p1 - __uint_as_float(u[i] & 0xFFFF0000u);
          }
        }
      };
      // P as packed bf16 pairs over the first 64 columns of S, or over P_t's own
      // columns with S prefetch (keys 2c, 2c+1 in column c); every S value is already
      // in registers.
      if constexpr (kSPrefetch) {
        const auto p_of_half = [&](int half, uint32_t (&u)[32]) { exp_half(half, u); };
        uint32_t u0[32], u1[32];
        p_of_half(0, u0);
        // P_t(j - 1) V(j - 1) must have read P_t (and finished adding into O_t) before
        // P_t is overwritten or O_t rescaled; the first half's exponentials above
        // overlap that product.
        if (step > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&bars.pv_done[t], (step - 1) & 1, &bars.abort, &g_fwd_status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        rescale_o();
        // The first half's store lands while the second half is computed; one wait
        // covers both before P_t is handed to the tensor core.
        tmem_st32_nowait(p_tm, u0);
        p_of_half(1, u1);
        tmem_st32_nowait(p_tm + 32, u1);
        tmem_wait_st();
      } else {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t u[32];
        exp_half(half, u);
        tmem_st32(p_tm + half * 32, u);
        if (!kPrecise && half == 0) {  // keys 0..63 are ready for the PV product
          tc_fence_before();
          mbar_arrive_warp(&bars.p_half[t]);
        }
      }
      }
      if (kPrecise) {  // residuals over columns 64..127 (the S values there are consumed)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t u[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = pack_bf16(x[half * 64 + 2 * i], x[half * 64 + 2 * i + 1]);
          tmem_st32(s_tm + 64 + half * 32, u);
        }
      }
      const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
      const float2 s4 = __fadd2_rn(s01, s23);
      const float rowsum = s4.x + s4.y;
      // Normaliser of O.  P enters the PV product rounded to bf16.  With the
      // reference max held back (lazy rescaling) the row's largest weight is
      // 2^(x_max - m) <= 2^32 instead of exactly 1, and its rounding error would
      // bias O by up to 2^-9 of a V row.  Adding that one element's rounding
      // error to the exact sum removes the bias; the other weights' rounding
      // errors are bounded and unbiased as in the standard bf16-P scheme.
      // (The same fused multiply-add and ex2 on the same input reproduce the
      // loop's value of that element bit for bit.)
      float delta_max = 0.f;
      if (!kPrecise) {
        const float p_max = ex2(fmaf(mx, sl2, neg_m));
        delta_max = __uint_as_float(pack_bf16(p_max, 0.f) << 16) - p_max;
      }
      l_run = l_run * alpha + rowsum;
      l_hat = kPrecise ? l_run : l_hat * alpha + (rowsum + delta_max);
      m_run = m_use;
      tc_fence_before();
      if (kPrecise) mbar_arrive_warp(&bars.p_half[t]);
      mbar_arrive_warp(&bars.p_full[t]);
    }
    // ------------------------------------------------------------ epilogue
    // The whole O row leaves tensor memory first; o_empty then lets the next item's
    // first P V product overwrite it while this row is normalised and stored.
    // O_t is complete once the item's last P V product is; with S prefetch that is
    // the tile's P V product before the step counter.  (The next item's first P V
    // product overwrites O_t: with S prefetch its issuer waits for this warp's first
    // P_t of that item, which comes after the loads below.)
    if (!ok || !__all_sync(0xffffffffu, kSPrefetch ? mbar_wait(&bars.pv_done[t], (step - 1) & 1, &bars.abort, &g_fwd_status)
                                                   : mbar_wait(&bars.o_full[t], it & 1, &bars.abort, &g_fwd_status))) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t orow[D];
#pragma unroll
    for (int c = 0; c < D; c += 64) {
      uint32_t (&part)[64] = *reinterpret_cast<uint32_t (*)[64]>(orow + c);
      tmem_ld64(o_tm + c, part);
    }
    tc_fence_before();
    if constexpr (!kSPrefetch) mbar_arrive_warp(&bars.o_empty[t]);
    {
      const float inv_l = 1.f / l_hat;
      const size_t row_off = (static_cast<size_t>(bh) * a.Nq + row) * D;
      const long long rows_total = static_cast<long long>(a.B) * a.H * a.Nq;
      // the row's D elements of O and its LSE lie inside [B, H, Nq, D] and [B, H, Nq]
      const bool store = row < a.Nq && in_bounds(static_cast<long long>(row_off) + D - 1, rows_total * D, &g_fwd_status) &&
                         in_bounds(static_cast<long long>(bh) * a.Nq + row, rows_total, &g_fwd_status);
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        const uint32_t* u = orow + c;
        if (store) {
          if (a.o_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.o) + row_off + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(u[4 * i]) * inv_l, __uint_as_float(u[4 * i + 1]) * inv_l,
                                   __uint_as_float(u[4 * i + 2]) * inv_l, __uint_as_float(u[4 * i + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + row_off + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(u[8 * i + e]) * inv_l;
              dst[i] = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                                  pack_bf16(f[6], f[7]));
            }
          }
        }
      }
      if (store) a.lse[static_cast<size_t>(bh) * a.Nq + row] = (m_run + __log2f(l_run)) * kLn2;
    }
    }
    if (a.stats != nullptr) {  // fa_set_stats counters: one addition per warp and CTA
      const unsigned resc = __reduce_add_sync(0xffffffffu, n_rescales);
      if (lane == 0 && resc != 0u) atomicAdd(a.stats + 2, static_cast<unsigned long long>(resc));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kPrecise>
cudaError_t launch_fwd_t(const ForwardArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, kPrecise>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split can only be granted from the registers the CTA is
  // launched with; refuse to launch rather than let the raise wait forever.
  cudaFuncAttributes attr{};
  e = cudaFuncGetAttributes(&attr, fwd_kernel<D, kPrecise>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * kFwdThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  const long long items = static_cast<long long>(a.B) * a.H * ((a.Nq + kBM * kTiles - 1) / (kBM * kTiles));
  if (items > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  // Persistent grid: one CTA per SM (each needs a whole SM's tensor memory), each
  // walking its share of the items.
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(items < sms ? items : sms));
  fwd_kernel<D, kPrecise><<<grid, kFwdThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, &g_fwd_status, limit_ns);  // nothing arrives
}

}  // namespace

cudaError_t launch_forward(const ForwardArgs& a, cudaStream_t stream) {
  if (a.d == 128) return a.precise ? launch_fwd_t<128, true>(a, stream) : launch_fwd_t<128, false>(a, stream);
  if (a.d == 64) return a.precise ? launch_fwd_t<64, true>(a, stream) : launch_fwd_t<64, false>(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_timeout_probe(unsigned long long limit_ns, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_clear_forward_status(unsigned* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fwd_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_fwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
