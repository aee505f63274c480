// Block-scaled grouped GEMMs of the a8w4 fused MoE layer on the sm_100-family
// 5th-generation tensor cores (tcgen05.mma kind::mxf8f6f4, TMEM accumulators,
// TMA + mbarrier pipeline), both stages:
//
//   stage 1: D[n, p] = sum_k W1[e][n, k] * X[p, k]    n over 2*Ip gate/up rows
//            epilogue: SiLU(gate)*up (no routing weight), per-1x32 FP8
//            requantisation of the intermediate (AITER #5609 "Add DeepSeek
//            V4.1 Flash TP4 gfx950 MoE tuning", Configuration)
//   stage 2: D[n, p] = sum_k W2[e][n, k] * A[p, k]    n over H features
//            epilogue: acc[token(p), n] += w_p * D[n, p] (FP32 reductions)
//
// The weights are the MMA's A operand (M = 128 weight rows per tile) and the
// routes its B operand (N = block_m routes), so a decode-sized expert group of
// a few routes costs an N=16 MMA instead of a mostly empty 128-row tile.
//
// Operand formats in shared memory (128-byte swizzled, K-major):
//   A  E2M1, prepacked in HBM as contiguous 8 KB tiles (128 rows x 64 bytes),
//      expanded by TMA (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B) to 16-byte
//      units holding 16 codes in their low 8 bytes, i.e. one byte slot per
//      element as kind::mxf8f6f4 expects for 4-bit operands; contiguous rows
//      stream at ~6 TB/s where 2560-byte-strided 64-byte rows reach ~4 TB/s;
//   B  E4M3 bytes.
// Scales: 512-byte atoms (128 rows x four 32-blocks, see sf_atom_off) copied
// to TMEM with tcgen05.cp .32x128b.warpx4 (4 columns per atom); the MMA for
// the i-th 32-block of a 128-K slab selects byte i of each 32-bit scale word.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner and
// MMA issuer, warps 2..5 = epilogue (TMEM lane quadrant = warp % 4).
// The kernel is persistent: CTA b walks tiles b, b + grid, ...; every role
// walks the same sequence and skips tiles past the device-side route count,
// so launch shapes depend only on host-known sizes (graph capturable).
#include <cstdint>
#include <cstring>
#include <type_traits>
#include <cuda.h>
#include <cudaTypedefs.h>
#include "common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "gemm_tiles.cuh"
#include "timeline.cuh"

MOE_TL_DEFINE(moe_tl_dump_mx)

namespace moe {
namespace {

#ifdef MOE_WAIT_STATS
// Experiment builds only: per-CTA cycles each role spent waiting on its
// barriers ([0] producer/empty, [1] MMA/full, [2] MMA/acc_empty,
// [3] epilogue/acc_full, [4] kernel cycles, [5] epilogue busy cycles).
__device__ long long g_wait_stats[512][16];   // [cta][(stage-1)*8 + slot]
#define WAIT_T0() const long long _wt0 = clock64()
#define WAIT_ADD(i) atomicAdd(reinterpret_cast<unsigned long long*>(&g_wait_stats[blockIdx.x][(a.stage - 1) * 8 + (i)]), \
                              static_cast<unsigned long long>(clock64() - _wt0))
#else
#define WAIT_T0()
#define WAIT_ADD(i)
#endif

constexpr int kThreads = 192;
constexpr int kTileN = 128;    // weight rows per tile (MMA M)
constexpr int kTileK = 128;    // K per pipeline stage
constexpr int kMmaK = 32;      // K per tcgen05.mma (8-bit slots)

struct MxArgs {
  int stage;             // 1 or 2
  int M, topk, H, Ip, E;
  int N, K;              // weight rows per expert / reduction length
  int n_tiles;           // N / 128
  int num_blocks;        // p_max / block_m
  int n_group_log2;      // stage 2: log2 of the feature tiles per walk group (-1: route-block major)
  int local;             // derive the route layout from topk_ids (decode sizes)
  const int32_t* topk_ids;
  LocalGate gate;        // gated calls: the routing input is the router logits
  const int32_t* sorted_route;
  const float* sorted_w;
  const int32_t* block_expert;
  const int32_t* num_padded;
  const uint8_t* w_base; // prepacked weight tiles [E][N/128][K/128][128][64 B]
  const uint8_t* sfa;    // weight scale atoms [E][N/128][K/128][512]
  const uint8_t* sfb;    // route scale atoms [blocks][K/128][na][512]
  uint8_t* inter;        // stage 1 out: E4M3 [p_max, Ip]
  uint8_t* inter_sf;     // stage 1 out: atoms [blocks][Ip/128][na][512]
  float* acc;            // stage 2 out: [M, H]
  int prefetch;          // weight L2 prefetch lead in k-blocks
  int32_t* status;
  // split walk, stage 1: FP32 partial sums [kSplitSlots][BN][128] and
  // arrival counters [kSplitSlots], zero at the start of the call
  float* split_part;
  int32_t* split_cnt;
};

template <int BN>
struct Cfg {
  static constexpr int kNa = (BN + 127) / 128;                 // scale atoms per B stage
  static constexpr int kABytes = kTileN * kTileK;              // 16 KB (expanded FP4)
  static constexpr int kBBytes = BN * kTileK;
  static constexpr int kSfBytes = 512 * (1 + kNa);
  static constexpr int kStageBytes = (kABytes + kBBytes + kSfBytes + 1023) / 1024 * 1024;
  // Up to block_m 64 two CTAs share an SM (two MMA-issuing threads: at small
  // N one thread cannot issue tcgen05 work fast enough to keep up with HBM),
  // so ring, accumulators and scale columns are sized for half an SM.
  // block_m 128 also runs two CTAs (single accumulator each: one CTA's
  // MMAs overlap the other's epilogue).
  static constexpr int kCtasPerSm = BN <= 128 ? 2 : 1;
  static constexpr int kStages = BN <= 16 ? 5 : BN <= 32 ? 4 : (BN <= 64 ? 4 : (BN <= 128 ? 3 : 4));
  static constexpr int kAccBufs = BN <= 64 ? 2 : 1;
  // Independent accumulators per tile: MMA kk of a k-block adds into
  // accumulator kk % kSplit, so small-N MMAs do not form one dependent chain;
  // the epilogue sums them.
  static constexpr int kSplit = BN <= 16 ? 2 : 1;
  static constexpr int kAccCols = BN * kSplit;
  static constexpr int kSfCols = 4 * (1 + kNa);                // TMEM columns per stage
  static constexpr int kColsNeeded = kAccBufs * kAccCols + kStages * kSfCols;
  static constexpr int kTmemCols = kColsNeeded <= 32 ? 32 : kColsNeeded <= 64 ? 64
                                   : kColsNeeded <= 128 ? 128 : kColsNeeded <= 256 ? 256 : 512;
  static constexpr int kEpiFloats = 32 * (64 + 4);             // stage-1 / stage-2 transpose tile
  static constexpr int kRouteBytes = BN * 8;                   // per-tile route info
  static constexpr int kSmem =
      1024 /*align slack*/ + kStages * kStageBytes + kEpiFloats * 4 + kRouteBytes + 256;
  // TMA transaction bytes of one stage: FP4 A counts packed bytes
  static constexpr uint32_t kTxBytes = kTileN * kTileK / 2 + kBBytes + kSfBytes;
  static_assert(kColsNeeded <= 512 / kCtasPerSm, "TMEM budget");
  // per SM: 228 KB of shared memory, of which 1 KB is reserved per CTA
  // per SM: 228 KB, of which 1 KB is reserved per CTA; the static shared
  // variables (barriers, the local route layout) take up to kStaticSmem
  static_assert(kCtasPerSm * (kSmem + 1024 + kStaticSmem) <= 228 * 1024, "smem budget");
};


template <int BN, bool SPLIT>
__global__ void __launch_bounds__(kThreads, Cfg<BN>::kCtasPerSm)
    moe_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const MxArgs a) {
  using C = Cfg<BN>;
  // SPLIT: the split walk (SplitSeq units; stage 1 finishes split tiles
  // through the partial-sum slots)
  // the producer's walk loads each tile's expert; the other roles' walks do not
  using Seq = typename std::conditional<SPLIT, SplitSeq<MxArgs>, TileSeq<MxArgs>>::type;
  using SeqR = typename std::conditional<SPLIT, SplitSeq<MxArgs, false>,
                                         TileSeq<MxArgs, false>>::type;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic so that the
  // compiler keeps every access below in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  float* epi = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  int* s_tok = reinterpret_cast<int*>(epi + C::kEpiFloats);      // [BN] token (stage 2) / -1 pad
  float* s_w = reinterpret_cast<float*>(s_tok + BN);              // [BN] routing weight
  __shared__ uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  __shared__ uint64_t acc_full[C::kAccBufs], acc_empty[C::kAccBufs];
  __shared__ uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int split_last;
  __shared__ uint16_t s_blk_expert[kLocalMaxBlocks];   // local layout: expert of each route block
  __shared__ int s_nblk;                               // local layout: number of route blocks

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) MOE_TL(3 + a.stage, 0);
  const int total_tiles = a.num_blocks * a.n_tiles;
  const int kblocks = a.K / kTileK;
#ifdef MOE_WAIT_STATS
  const long long _k0 = clock64();
#endif

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // Decode sizes: the route layout (route blocks per expert) is derived here
  // from topk_ids, an input of the call that is complete before the call's
  // first kernel starts, so the producer can load its first weight tiles
  // before the previous kernel has finished (see LocalLayout).
  if (a.local) {
    // the epilogue's transpose buffer is free until the first tile's epilogue
    const int nb = local_block_layout(a.topk_ids, a.M * a.topk, a.E, BN,
                                      reinterpret_cast<int*>(epi), s_blk_expert, a.gate, a.M);
    if (threadIdx.x == 0) s_nblk = nb;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sf_col0 = C::kAccBufs * C::kAccCols;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per tile the weight tiles (prepacked: consecutive k-blocks are
    // consecutive 8 KB blocks), both scale arrays and the route rows advance
    // by constant steps. A second cursor runs kPrefetch k-blocks ahead
    // (across tiles) and prefetches weight tiles into L2, so the loads that
    // fill the shared-memory ring mostly hit L2. With the local layout the
    // weight half of the first ring stages (weights and their scales) is
    // loaded before the dependency wait and the route half after it.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();   // weights: streamed once
      const uint64_t pol_x = policy_evict_last();    // routes: reused across n-tiles
      // k-blocks the L2 prefetch runs ahead (per call; the defaults are set
      // where the launch is prepared)
      const int kPrefetch = a.prefetch;
      constexpr uint32_t kWTile = kTileN * kTileK / 2;   // 8 KB
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_mask = 0, armed_par = 0;   // stages armed, parity of their last arming
      uint8_t* sbase = stages;
#ifdef MOE_TIMELINE
      int tl_first = 1;
#endif
      auto produce = [&](auto cur, auto expert_of, auto local_mode) {
        constexpr bool kLocal = decltype(local_mode)::value;
        int P;
        if constexpr (kLocal) {
          P = s_nblk * BN;
        } else {
          pdl_wait_prior();
          if (threadIdx.x == 0) MOE_TL(3 + a.stage, 1);
          P = *a.num_padded;
        }
        seq_init(cur, a, total_tiles, P, BN, kblocks);
        auto pf = cur;
        int pf_kb = 0;
        const uint8_t* pf_w = nullptr;
        auto pf_tile = [&]() {
          pf_w = a.w_base + (static_cast<int64_t>(expert_of(pf)) * a.n_tiles + pf.n_tile) *
                                kblocks * kWTile;
          pf_kb = seq_kb0(pf);
        };
        if (pf.valid) pf_tile();
        auto pf_skip = [&]() {
          if (++pf_kb == seq_kb1(pf, kblocks)) {
            seq_next(pf, a, total_tiles, P, BN);
            if (pf.valid) pf_tile();
          }
        };
        auto pf_step = [&]() {
          if (!pf.valid) return;
          bulk_prefetch_l2(pf_w + static_cast<int64_t>(pf_kb) * kWTile, kWTile);
          pf_skip();
        };
        // flat walk over the k-blocks of this CTA's tiles
        int kb = 0, kb_end = 0, row_a = 0, row_b = 0;
        const uint8_t* sfa = nullptr;
        const uint8_t* sfb = nullptr;
        auto set_tile = [&]() {
          const int64_t wtile = static_cast<int64_t>(expert_of(cur)) * a.n_tiles + cur.n_tile;
          kb = seq_kb0(cur);
          kb_end = seq_kb1(cur, kblocks);
          row_a = static_cast<int>((wtile * kblocks + kb) * kTileN);
          sfa = a.sfa + (wtile * kblocks + kb) * 512;
          sfb = a.sfb + (static_cast<int64_t>(cur.m_blk) * kblocks + kb) * C::kNa * 512;
          row_b = cur.m_blk * BN;
        };
        auto advance = [&](bool prefetch) {
          if (prefetch) pf_step();
          else if (pf.valid) pf_skip();
          row_a += kTileN;
          sfa += 512;
          sfb += 512 * C::kNa;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
            sbase = stages;
          } else {
            sbase += C::kStageBytes;
          }
          if (++kb == kb_end) {
            seq_next(cur, a, total_tiles, P, BN);
            if (cur.valid) set_tile();
          }
        };
        auto arm = [&]() {
          mbar_arrive_expect_tx(&full_bar[stage], C::kTxBytes);
          armed_mask |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
#ifdef MOE_TIMELINE
          if (tl_first) { MOE_TL(3 + a.stage, 2); tl_first = 0; }
#endif
        };
        auto load_w = [&]() {
          tma_load_2d(sbase, &tmA, &full_bar[stage], 0, row_a, pol_w);
          bulk_load(sbase + C::kABytes + C::kBBytes, sfa, 512, &full_bar[stage], pol_w);
        };
        auto load_x = [&](uint8_t* sb, uint64_t* bar, int kbx, int rb, const uint8_t* sfbx) {
          tma_load_2d(sb + C::kABytes, &tmB, bar, kbx * kTileK, rb, pol_x);
          bulk_load(sb + C::kABytes + C::kBBytes + 512, sfbx, 512 * C::kNa, bar, pol_x);
        };
        if (cur.valid) set_tile();
        // The L2 prefetch cursor runs kPrefetch k-blocks ahead of the loads.
        // With the local layout its first burst is issued after the copies
        // of the preloaded stages, before the dependency wait (measured: this
        // order beat a burst after the wait and a burst from another thread).
        if constexpr (!kLocal) {
          for (int i = 0; i < kPrefetch; ++i) pf_step();
        }
        if constexpr (kLocal) {
          // the first ring stages: weights now, routes after the wait
          int npre = 0;
          int pre_kb[C::kStages], pre_rb[C::kStages];
          const uint8_t* pre_sfb[C::kStages];
          while (cur.valid && npre < C::kStages) {
            arm();
            load_w();
            pre_kb[npre] = kb;
            pre_rb[npre] = row_b;
            pre_sfb[npre] = sfb;
            ++npre;
            advance(false);   // these k-blocks are being loaded, not prefetched
          }
          for (int i = 0; i < kPrefetch; ++i) pf_step();
          pdl_wait_prior();
          if (threadIdx.x == 0) MOE_TL(3 + a.stage, 1);
          for (int i = 0; i < npre; ++i)
            load_x(stages + i * C::kStageBytes, &full_bar[i], pre_kb[i], pre_rb[i], pre_sfb[i]);
        }
        while (cur.valid && !abort_flag) {
          {
            WAIT_T0();
            if (!mbar_wait(&empty_bar[stage], phase ^ 1, a.status)) { abort_flag = 1; break; }
            WAIT_ADD(0);
          }
          arm();
          load_w();
          load_x(sbase, &full_bar[stage], kb, row_b, sfb);
          advance(true);
        }
        if constexpr (kLocal) {
          // the layout derived from topk_ids must be the sort's
          if (*a.num_padded != P && a.status) atomicOr(a.status, kDevBadExpert);
        }
      };
      if (a.local)
        produce(SeqR{}, [&](const SeqR& q) { return static_cast<int>(s_blk_expert[q.m_blk]); },
                std::true_type{});
      else
        produce(Seq{}, [](const Seq& q) { return q.e; }, std::false_type{});
      // Copies still in flight into shared memory must land before the CTA
      // exits: normally the MMA thread consumed every armed stage, so these
      // return at once; after an abort they wait (bounded) for the TMA.
      for (int s = 0; s < C::kStages; ++s)
        if ((armed_mask >> s) & 1u) mbar_wait(&full_bar[s], (armed_par >> s) & 1u, a.status);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    // At small N the tensor core is far faster than one thread can issue, so
    // this loop is kept minimal: descriptors are built once and advanced by
    // adding to their 14-bit start-address field (address >> 4), instruction
    // descriptors are compile-time constants.
    pdl_wait_prior();
    const int P = a.local ? s_nblk * BN : *a.num_padded;
    if (lane == 0) {
      const uint64_t a_desc0 = smem_desc(smem_u32(stages), 16, 1024, kSwizzle128B);
      const uint64_t b_desc0 = smem_desc(smem_u32(stages + C::kABytes), 16, 1024, kSwizzle128B);
      const uint64_t sf_desc0 = smem_desc(smem_u32(stages + C::kABytes + C::kBBytes), 0, 128,
                                          kSwizzleNone);
      constexpr uint32_t kStageStep = C::kStageBytes >> 4;   // descriptor units per stage
      int stage = 0;
      uint32_t phase = 0;
      uint32_t sdesc_off = 0;                                // stage * kStageStep
      uint32_t sf_tmem = tmem + sf_col0;                      // this stage's scale columns
      int local = 0;
      SeqR seq;
#ifdef MOE_TIMELINE
      int tl_mma = 1;
#endif
      for (seq_init(seq, a, total_tiles, P, BN, kblocks); seq.valid && !abort_flag;
           seq_next(seq, a, total_tiles, P, BN)) {
        const int ab = local % C::kAccBufs;
        const uint32_t acc_phase = (local / C::kAccBufs) & 1;
        ++local;
        {
          WAIT_T0();
          if (!mbar_wait(&acc_empty[ab], acc_phase ^ 1, a.status)) { abort_flag = 1; break; }
          WAIT_ADD(2);
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + ab * C::kAccCols;
        const int kb_begin = seq_kb0(seq), kb_end = seq_kb1(seq, kblocks);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          {
            WAIT_T0();
            if (!mbar_wait(&full_bar[stage], phase, a.status)) { abort_flag = 1; break; }
            WAIT_ADD(1);
          }
#ifdef MOE_TIMELINE
          if (tl_mma) { MOE_TL(3 + a.stage, 3); tl_mma = 0; }
#endif
          tmem_cp_32x128b_warpx4(sf_tmem, sf_desc0 + sdesc_off);
#pragma unroll
          for (int j = 0; j < C::kNa; ++j)
            tmem_cp_32x128b_warpx4(sf_tmem + 4 + 4 * j, sf_desc0 + sdesc_off + 32 * (1 + j));
          const uint64_t ad = a_desc0 + sdesc_off;
          const uint64_t bd = b_desc0 + sdesc_off;
#pragma unroll
          for (int kk = 0; kk < kTileK / kMmaK; ++kk) {
            mma_mxf8f6f4(d_tmem + (kk % C::kSplit) * BN, ad + 2 * kk, bd + 2 * kk,
                         idesc_mx(5, 0, kTileN, BN, kk, kk), sf_tmem, sf_tmem + 4,
                         kb > kb_begin || kk >= C::kSplit);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
            sdesc_off = 0;
            sf_tmem = tmem + sf_col0;
          } else {
            sdesc_off += kStageStep;
            sf_tmem += C::kSfCols;
          }
        }
        tc_commit(&acc_full[ab]);
      }
      // every MMA issued by this thread has finished before TMEM is released
      MOE_TL(3 + a.stage, 4);
      tc_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, a.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait_prior();
    const int P = a.local ? s_nblk * BN : *a.num_padded;
    const int quad = warp & 3;               // TMEM lane quadrant
    const int row = quad * 32 + lane;        // weight row within the tile
    const int et = threadIdx.x - 64;         // 0..127
    const int R = a.M * a.topk;
    int local = 0;
    SeqR seq;
    for (seq_init(seq, a, total_tiles, P, BN, kblocks); seq.valid;
         seq_next(seq, a, total_tiles, P, BN)) {
      const int m_blk = seq.m_blk, n_tile = seq.n_tile;
      const int ab = local % C::kAccBufs;
      const uint32_t acc_phase = (local / C::kAccBufs) & 1;
      ++local;
      // Route info of the tile's columns (token or -1 for a pad, weight),
      // loaded before waiting for the accumulator.
      {
        const int64_t pb = static_cast<int64_t>(m_blk) * BN;
        named_bar_sync(1, 128);               // previous tile's readers are done
        for (int c = et; c < BN; c += 128) {
          const int rr = __ldg(a.sorted_route + pb + c);
          const int tok = rr < R ? rr / a.topk : -1;
          s_tok[c] = tok;
          s_w[c] = __ldg(a.sorted_w + pb + c);
        }
        named_bar_sync(1, 128);
      }
      {
        WAIT_T0();
        if (abort_flag || !mbar_wait(&acc_full[ab], acc_phase, a.status)) { abort_flag = 1; break; }
        if (threadIdx.x == 64) WAIT_ADD(3);
      }
#ifdef MOE_WAIT_STATS
      const long long _busy0 = clock64();
#endif
      tc_fence_after();
      const uint32_t d_tmem = tmem + ab * C::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
      const int64_t p_base = static_cast<int64_t>(m_blk) * BN;
      constexpr int kChunk = BN < 32 ? BN : 32;
      // Split walk, stage 1: a part of a split tile adds its partial sums to
      // the tile's slot (feature row fastest: a warp adds 128 contiguous
      // bytes), releases the accumulator and counts itself in; the part that
      // arrives last reads the complete sums back from L2 and runs the
      // epilogue. (Stage 2 adds every part to the accumulator directly.)
      float* part = nullptr;
      if constexpr (SPLIT) {
        if (seq.slot >= 0 && a.stage == 1) {
          part = a.split_part + static_cast<int64_t>(seq.slot) * BN * 128;
          for (int c0 = 0; c0 < BN; c0 += kChunk) {
            float v[32];
#pragma unroll
            for (int sp = 0; sp < C::kSplit; ++sp) {
              uint32_t r[32];
              if constexpr (kChunk == 32) {
                tmem_ld_32x32b_x32(d_tmem + sp * BN + c0, r);
              } else {
                uint32_t r16[16];
                tmem_ld_32x32b_x16(d_tmem + sp * BN + c0, r16);
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = r16[i];
              }
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < kChunk; ++i)
                v[i] = sp == 0 ? __uint_as_float(r[i]) : v[i] + __uint_as_float(r[i]);
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) atomicAdd(part + (c0 + i) * 128 + row, v[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[ab]);
          __threadfence();
          named_bar_sync(1, 128);
          if (et == 0) split_last = atomicAdd(a.split_cnt + seq.slot, 1) == seq.parts - 1;
          named_bar_sync(1, 128);
          if (!split_last) continue;
          __threadfence();
        }
      }
      // The chunk's epilogue once its FP32 values are in v (from TMEM, or
      // from the split slot for the last part of a split stage-1 tile). The
      // two loops below keep the TMEM path free of the slot pointer: with
      // it in one loop the split kernel's stage 2 ran 2x slower.
      auto finish = [&](const int c0, float (&v)[32]) {
        if (a.stage == 1) {
          // Gate (row 2j) and up (row 2j+1) sit in adjacent lanes. Even lanes
          // produce columns [0, half), odd lanes [half, kChunk): one shuffle
          // per column pair, no divergence.
          constexpr int half = kChunk / 2;
          const bool odd = lane & 1;
          const int j_local = row >> 1;       // 0..63
          named_bar_sync(1, 128);             // previous chunk's readers are done
#pragma unroll
          for (int k = 0; k < half; ++k) {
            const float send = odd ? v[k] : v[k + half];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float gate = odd ? recv : v[k];
            const float up = odd ? v[k + half] : recv;
            epi[(k + (odd ? half : 0)) * 68 + j_local] = __fdividef(gate, 1.0f + __expf(-gate)) * up;
          }
          named_bar_sync(1, 128);
          // 2 threads per (route column, 32-block): each quantises 16 values
          const int item = et >> 1, hf = et & 1;       // 64 items
          const int col = item >> 1, blk = item & 1;   // column in chunk, 32-block in tile
          if (col < kChunk) {
            const int64_t p = p_base + c0 + col;
            const bool pad = s_tok[c0 + col] < 0;
            float x[16];
            const float4* src = reinterpret_cast<const float4*>(epi + col * 68 + blk * 32 + hf * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 f = src[q];
              x[4 * q] = f.x; x[4 * q + 1] = f.y; x[4 * q + 2] = f.z; x[4 * q + 3] = f.w;
            }
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            if (pad) amax = 0.f;
            uint32_t codes[4] = {0u, 0u, 0u, 0u};
            int sb = 0;
            if (amax != 0.f) {
              sb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 8;
              sb = sb < 0 ? 0 : sb;
              const float inv = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(x[4 * i] * inv, x[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(x[4 * i + 2] * inv, x[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
                codes[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
              }
            }
            const int jcol = n_tile * 64 + blk * 32 + hf * 16;     // intermediate column
            *reinterpret_cast<uint4*>(a.inter + p * a.Ip + jcol) =
                make_uint4(codes[0], codes[1], codes[2], codes[3]);
            if (hf == 0) {
              const int ib = jcol / 32;                          // 32-block index along Ip
              const int rr = c0 + col;                           // row of p inside the block
              const int64_t atom = (static_cast<int64_t>(m_blk) * (a.Ip / 128) + ib / 4) * C::kNa + rr / 128;
              a.inter_sf[atom * 512 + sf_atom_off(rr & 127, ib & 3)] = static_cast<uint8_t>(sb);
            }
          }
        } else if constexpr (BN >= 64) {
          // stage 2, large tiles: the chunk's weighted values go through
          // shared memory route-major (8 routes x 128 features per pass, two
          // alternating buffers, one barrier per pass), and each warp then adds
          // whole 512-byte token-row segments with 16-byte vector reductions:
          // a quarter of the reduction instructions of the register path.
          const int64_t col0 = static_cast<int64_t>(n_tile) * kTileN + 4 * lane;
#pragma unroll
          for (int h = 0; h < kChunk / 8; ++h) {
            float* buf = epi + (h & 1) * (8 * kTileN);
            const float4 wa = reinterpret_cast<const float4*>(s_w + c0 + h * 8)[0];
            const float4 wb = reinterpret_cast<const float4*>(s_w + c0 + h * 8)[1];
            const float wk[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) buf[i * kTileN + row] = v[h * 8 + i] * wk[i];
            named_bar_sync(1, 128);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int r = quad * 2 + j;
              const int tok = s_tok[c0 + h * 8 + r];
              if (tok < 0) continue;
              const float4 f = reinterpret_cast<const float4*>(buf + r * kTileN)[lane];
              atomicAdd(reinterpret_cast<float4*>(a.acc + static_cast<int64_t>(tok) * a.H + col0), f);
            }
          }
        } else {
          // stage 2: this thread holds output feature `row` of the tile for
          // the chunk's routes, so a warp adds 32 consecutive features (128
          // contiguous bytes of one token row) per reduction, from registers;
          // the route info is read four routes per 16-byte broadcast load
          float* col = a.acc + static_cast<int64_t>(n_tile) * kTileN + row;
#pragma unroll
          for (int q = 0; q < kChunk / 4; ++q) {
            const int4 t4 = reinterpret_cast<const int4*>(s_tok + c0)[q];
            const float4 w4 = reinterpret_cast<const float4*>(s_w + c0)[q];
            const int tk[4] = {t4.x, t4.y, t4.z, t4.w};
            const float wk[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (tk[j] >= 0) atomicAdd(col + static_cast<int64_t>(tk[j]) * a.H, v[4 * q + j] * wk[j]);
          }
        }
      };
      if (SPLIT && part) {
        for (int c0 = 0; c0 < BN; c0 += kChunk) {
          float v[32];
#pragma unroll
          for (int i = 0; i < kChunk; ++i) v[i] = __ldcg(part + (c0 + i) * 128 + row);
          finish(c0, v);
        }
      } else {
        for (int c0 = 0; c0 < BN; c0 += kChunk) {
          float v[32];
#pragma unroll
          for (int sp = 0; sp < C::kSplit; ++sp) {
            uint32_t r[32];
            if constexpr (kChunk == 32) {
              tmem_ld_32x32b_x32(d_tmem + sp * BN + c0, r);
            } else {
              uint32_t r16[16];
              tmem_ld_32x32b_x16(d_tmem + sp * BN + c0, r16);
#pragma unroll
              for (int i = 0; i < 16; ++i) r[i] = r16[i];
            }
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < kChunk; ++i)
              v[i] = sp == 0 ? __uint_as_float(r[i]) : v[i] + __uint_as_float(r[i]);
          }
          finish(c0, v);
        }
      }
      if (!SPLIT || !part) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
      }
#ifdef MOE_WAIT_STATS
      if (threadIdx.x == 64)
        atomicAdd(reinterpret_cast<unsigned long long*>(&g_wait_stats[blockIdx.x][(a.stage - 1) * 8 + 5]),
                  static_cast<unsigned long long>(clock64() - _busy0));
#endif
    }
    if (threadIdx.x == 64) MOE_TL(3 + a.stage, 5);
    if (a.stage == 1) {
      // Zero this CTA's share of the FP32 accumulator that stage 2 reduces
      // into, after this CTA's last tile: at decode sizes the lines are then
      // still in L2 when stage 2 starts (which waits for this grid).
      const int64_t n4 = static_cast<int64_t>(a.M) * a.H / 4;
      const int64_t per = (n4 + gridDim.x - 1) / gridDim.x;
      const int64_t lo = static_cast<int64_t>(blockIdx.x) * per;
      const int64_t hi = lo + per < n4 ? lo + per : n4;
      float4* a4 = reinterpret_cast<float4*>(a.acc);
      for (int64_t i = lo + et; i < hi; i += 128) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    MOE_TL(3 + a.stage, 7);
  }
#ifdef MOE_WAIT_STATS
  if (threadIdx.x == 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(&g_wait_stats[blockIdx.x][(a.stage - 1) * 8 + 4]),
              static_cast<unsigned long long>(clock64() - _k0));
#endif
}

}  // namespace

#ifdef MOE_WAIT_STATS
extern "C" void moe_debug_wait_stats(long long* host_out, int reset) {
  cudaMemcpyFromSymbol(host_out, g_wait_stats, sizeof(g_wait_stats));
  if (reset) {
    static long long zeros[512][16] = {};
    cudaMemcpyToSymbol(g_wait_stats, zeros, sizeof(zeros));
  }
}
#endif

namespace {

// ---------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
               uint64_t rows, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t plan_bn(const MxArgs& a, int split, int num_sms, GemmPlan* plan) {
  using C = Cfg<BN>;
  static_assert(sizeof(MxArgs) <= sizeof(plan->args), "argument block");
  // The split-walk kernel at route blocks <= 32 unless the call asks for
  // whole tiles (split = 2): it splits where the real tiles are fewer than
  // kSplitMaxWaves waves and otherwise walks whole tiles route-block major,
  // measured as fast as the plain kernel or faster at every decode size but
  // the draft geometry's 10-20 tokens (up to 5 % faster at 192-768 tokens).
  // Stage 1 needs the split slots of the workspace.
  const void* fn = reinterpret_cast<const void*>(&moe_gemm_mx_kernel<BN, false>);
  if constexpr (BN <= 32) {
    if (split != 2 && (a.stage == 2 || a.split_part))
      fn = reinterpret_cast<const void*>(&moe_gemm_mx_kernel<BN, true>);
  }
  cudaError_t err = ensure_smem_attr(fn, C::kSmem);
  if (err != cudaSuccess) return err;
  const int tiles = a.num_blocks * a.n_tiles;
  const int slots = num_sms * C::kCtasPerSm;
  plan->kernel = fn;
  // the split kernel spreads the k-blocks over every CTA slot
  const bool split_kernel = fn != reinterpret_cast<const void*>(&moe_gemm_mx_kernel<BN, false>);
  plan->grid = split_kernel || tiles > slots ? slots : tiles;
  plan->threads = kThreads;
  plan->smem = C::kSmem;
  memcpy(plan->args, &a, sizeof(a));
  return cudaSuccess;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

}  // namespace

cudaError_t prepare_gemm_mx(int stage, const GemmArgs& g, GemmPlan* plan) {
  MxArgs a{};
  a.stage = stage;
  a.M = g.M; a.topk = g.topk; a.H = g.H; a.Ip = g.Ip; a.E = g.E;
  a.N = stage == 1 ? 2 * g.Ip : g.H;
  a.K = stage == 1 ? g.H : g.Ip;
  a.n_tiles = a.N / kTileN;
  a.num_blocks = static_cast<int>(g.p_max / g.bm);
  a.n_group_log2 = stage == 1 ? 0 : stage2_n_group_log2(g.M, g.p_max * g.Ip * 1, a.n_tiles);
  a.local = (g.topk_ids || g.gate.logits) &&
            static_cast<int64_t>(g.M) * g.topk <= kLocalMaxRoutes &&
            a.num_blocks <= kLocalMaxBlocks ? 1 : 0;
  a.topk_ids = g.topk_ids;
  a.gate = g.gate;
  a.sorted_route = g.sorted_route; a.sorted_w = g.sorted_w; a.block_expert = g.block_expert;
  a.num_padded = g.num_padded;
  a.sfa = stage == 1 ? g.w1s : g.w2s;
  a.w_base = stage == 1 ? g.w1 : g.w2;
  a.sfb = stage == 1 ? g.act_sf : g.inter_sf;
  a.inter = static_cast<uint8_t*>(g.inter);
  a.inter_sf = g.inter_sf;
  a.acc = g.acc;
  // default leads 4 and 2 tiles: the tuned decode rows of every a8w4
  // geometry settled on them (1-10 % faster than 16 / 8) and they are also
  // the fastest measured at prefill (M=4096-16384: 0.5-1.3 %; 32 or 64 tiles
  // are slower)
  a.prefetch = stage == 1 ? (g.prefetch1 > 0 ? g.prefetch1 : 4)
                         : (g.prefetch2 > 0 ? g.prefetch2 : 2);
  a.status = g.status;
  a.split_part = g.split_part;
  a.split_cnt = g.split_cnt;
  plan->grid = 0;
  if (a.num_blocks == 0) return cudaSuccess;
  const uint8_t* w = stage == 1 ? g.w1 : g.w2;
  const void* xb = stage == 1 ? g.act : g.inter;
  CUtensorMap* ta = reinterpret_cast<CUtensorMap*>(plan->tmap_a);
  CUtensorMap* tb = reinterpret_cast<CUtensorMap*>(plan->tmap_b);
  if (!encode_2d(ta, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, kTileK,
                 static_cast<uint64_t>(a.E) * a.N * (a.K / kTileK), kTileK / 2, kTileK, kTileN))
    return cudaErrorInvalidValue;
  if (!encode_2d(tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, xb, a.K, static_cast<uint64_t>(g.p_max), a.K,
                 128, g.bm))
    return cudaErrorInvalidValue;
  const int sms = sm_count();
  switch (g.bm) {
    case 16: return plan_bn<16>(a, g.split, sms, plan);
    case 32: return plan_bn<32>(a, g.split, sms, plan);
    case 64: return plan_bn<64>(a, g.split, sms, plan);
    case 128: return plan_bn<128>(a, g.split, sms, plan);
    case 256: return plan_bn<256>(a, g.split, sms, plan);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(const GemmPlan& plan, cudaStream_t s) {
  if (plan.grid <= 0) return cudaSuccess;
  void* args[3] = {const_cast<unsigned char*>(plan.tmap_a), const_cast<unsigned char*>(plan.tmap_b),
                   const_cast<unsigned char*>(plan.args)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(plan.threads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, plan.kernel, args);
}

}  // namespace moe
