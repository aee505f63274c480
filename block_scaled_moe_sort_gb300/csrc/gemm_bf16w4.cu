// Grouped GEMMs of the a16w4 fused MoE layer (BF16 activations x MXFP4
// weights; AITER #6286 "Retune gfx942 a16w4 DSv4.1 tiles for Triton 3.8",
// reviewer reply: moe_gemm_a16w4 with w1 apply_swiglu=True, w2 separate,
// bf16, MXFP4) on tcgen05.mma kind::f16 with TMEM accumulators:
//
//   stage 1: D[n, p] = sum_k W1[e][n, k] * X[p, k]; epilogue SiLU(gate)*up,
//            rounded to a BF16 intermediate
//   stage 2: D[n, p] = sum_k W2[e][n, k] * A[p, k]; epilogue
//            acc[token(p), n] += w_p * D[n, p]
//
// kind::f16 needs both operands in the same 16-bit type, so the MXFP4
// weights are dequantised on chip: every E2M1 value times its E8M0 scale is
// a BF16 number (exact: a 2-bit-mantissa value times a power of two), so the
// MMA sees exactly the weights the format encodes. The dequantised weight
// tile never touches shared memory: converter threads write it straight into
// TMEM (one weight row per TMEM lane) and the MMA reads its A operand from
// there, so a shared-memory stage holds only the packed FP4 tile, its scales
// and the activation rows, and the ring can be deep.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps
// 2..5 epilogue (TMEM lane quadrant = warp % 4), warps 6.. converters (4 or
// 8; quadrant = warp % 4, with 8 warps each converts half of the stage's K).
// A converter thread turns its row's FP4 pairs into BF16 pairs with
// rotations and masks (the a16w4 weight prepack stores every word in the bit
// order that makes this work, dequant_a16.cuh), multiplies by the block
// scale and stores 32 TMEM columns at a time; no lookup table, so shared
// memory bandwidth stays with the TMA and the MMA's B operand.
// Pipeline stage = 128 K-elements: one prepacked 8 KB weight tile, fetched by
// TMA with the 64-byte swizzle (conflict-free row reads), its 512-byte scale
// atom, and two 128-byte swizzle atoms of BF16 activations.
#include <cstdint>
#include <cstring>
#include <type_traits>
#include <cuda.h>
#include <cudaTypedefs.h>
#include "common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "gemm_tiles.cuh"
#include "dequant_a16.cuh"
#include "timeline.cuh"

MOE_TL_DEFINE(moe_tl_dump_bf16)

namespace moe {
namespace {

#ifdef MOE_WAIT_STATS
// Experiment builds only: per-CTA cycles each role spent at its barriers,
// [cta][stage-1][slot]: 0 producer/empty, 1 MMA/full, 2 MMA/a_full,
// 3 MMA/acc_empty, 4 converter/full, 5 converter/a_empty, 6 converter busy,
// 7 epilogue/acc_full, 8 kernel cycles.
__device__ long long g_ws16[512][2][16];
#define WS_T0() const long long _wt0 = clock64()
#define WS_ADD(i) atomicAdd(reinterpret_cast<unsigned long long*>(&g_ws16[blockIdx.x & 511][a.stage - 1][(i)]), \
                            static_cast<unsigned long long>(clock64() - _wt0))
#else
#define WS_T0()
#define WS_ADD(i)
#endif

constexpr int kTileN = 128;   // weight rows per tile (MMA M)
constexpr int kTileK = 128;   // K per stage = one prepacked 8 KB weight tile
constexpr int kMmaK = 16;     // K per tcgen05.mma kind::f16
constexpr int kAtomK = 64;    // BF16 elements per 128-byte swizzle atom row
constexpr int kACols = 64;    // TMEM columns of one dequantised 128 x 128 BF16 tile

struct Bf16Args {
  int stage;
  int M, topk, H, Ip, E;
  int N, K;
  int n_tiles;
  int num_blocks;
  int n_group_log2;            // stage 2: log2 of the feature tiles per walk group (-1: route-block major)
  int local;                   // derive the route layout from topk_ids (decode sizes)
  const int32_t* topk_ids;
  LocalGate gate;        // gated calls: the routing input is the router logits
  const int32_t* sorted_route;
  const float* sorted_w;
  const int32_t* block_expert;
  const int32_t* num_padded;
  const uint8_t* w;            // prepacked E2M1 tiles [E][N/128][K/128][128][64 B]
  const uint8_t* sfa;          // weight scale atoms [E][N/128][K/128][512]
  __nv_bfloat16* inter;        // stage 1 out: BF16 [p_max, Ip]
  float* acc;                  // stage 2 out
  int prefetch;                // weight L2 prefetch lead in k-blocks
  int32_t* status;
  // split walk, stage 1: FP32 partial sums [kSplitSlots][BN][128] and
  // arrival counters [kSplitSlots], zero at the start of the call
  float* split_part;
  int32_t* split_cnt;
};

__host__ __device__ constexpr int pow2_cols(int c) {
  return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512;
}

template <int BN>
struct Cfg16 {
  // Small route blocks run two CTAs per SM so that two MMA issuers and two
  // converter groups share the SM. Shared-memory stages (the TMA ring) and
  // TMEM slots of dequantised weight tiles are two rings of their own
  // depths: k-block j uses stage j % kStages and slot j % kASlots. The MMA's
  // one commit per k-block frees both its stage and its slot; the converter
  // writes slot j % kASlots once the stage of k-block j has landed and the
  // MMA of k-block j - kASlots has committed. TMEM bounds the slots (3 at
  // two CTAs per SM); shared memory bounds the stages, so at small route
  // blocks the TMA runs up to kStages k-blocks ahead while the converters run
  // up to kASlots ahead of the MMA.
  static constexpr int kCtasPerSm = BN <= 32 ? 2 : 1;
  static constexpr int kConvWarps = kCtasPerSm == 2 ? 4 : 8;
  static constexpr int kThreads = 192 + 32 * kConvWarps;
  static constexpr int kRawBytes = kTileN * kTileK / 2;        // 8 KB packed FP4
  static constexpr int kSfBytes = 512;
  static constexpr int kBAtomBytes = BN * 128;                 // BN rows x 64 BF16
  static constexpr int kBBytes = 2 * kBAtomBytes;
  // stage layout: B atoms, raw FP4 tile (64-byte swizzled), scale atom
  static constexpr int kStageBytes = (kBBytes + kRawBytes + kSfBytes + 1023) / 1024 * 1024;
  static constexpr int kASlots = BN <= 32 ? 3 : BN == 64 ? 6 : BN == 128 ? 4 : 2;
  static constexpr int kStages = kASlots;
  static_assert(kStages >= kASlots, "a slot is reused only after its stage was");
  static constexpr int kAccBufs = BN <= 128 ? 2 : 1;
  static constexpr int kAccCol0 = kASlots * kACols;
  static constexpr int kTmemCols = pow2_cols(kAccCol0 + kAccBufs * BN);
  static constexpr int kEpiFloats = 32 * (64 + 4);
  static constexpr int kRouteBytes = BN * 8;                   // per-tile route info
  static constexpr int kSmem =
      1024 + kStages * kStageBytes + kEpiFloats * 4 + kRouteBytes;
  static constexpr uint32_t kTxBytes = kRawBytes + kSfBytes + kBBytes;
  // per SM: 228 KB, of which 1 KB is reserved per CTA; the static shared
  // variables (barriers, the local route layout) take up to kStaticSmem
  static_assert(kCtasPerSm * (kSmem + 1024 + kStaticSmem) <= 228 * 1024, "smem budget");
  static_assert(kAccCol0 + kAccBufs * BN <= kTmemCols && kTmemCols * kCtasPerSm <= 512,
                "TMEM budget");
};

// SPLIT: the split walk (SplitSeq units; stage 1 finishes split tiles
// through the partial-sum slots), else whole tiles (TileSeq)
template <int BN, bool SPLIT>
__global__ void __launch_bounds__(Cfg16<BN>::kThreads, Cfg16<BN>::kCtasPerSm)
    moe_gemm_bf16w4_kernel(const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmX, const Bf16Args a) {
  using C = Cfg16<BN>;
  // the producer's walk loads each tile's expert; the other roles' walks do not
  using Seq16 = typename std::conditional<SPLIT, SplitSeq<Bf16Args>, TileSeq<Bf16Args>>::type;
  using Seq16R = typename std::conditional<SPLIT, SplitSeq<Bf16Args, false>,
                                           TileSeq<Bf16Args, false>>::type;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic so that the
  // compiler keeps every access below in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* epi = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  int* s_tok = reinterpret_cast<int*>(epi + C::kEpiFloats);      // [BN] token / -1 pad
  float* s_w = reinterpret_cast<float*>(s_tok + BN);              // [BN] routing weight
  __shared__ uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  __shared__ uint64_t a_full[C::kASlots];
  __shared__ uint64_t acc_full[C::kAccBufs], acc_empty[C::kAccBufs];
  __shared__ uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int split_last;
  __shared__ uint16_t s_blk_expert[kLocalMaxBlocks];   // local layout: expert of each route block
  __shared__ int s_nblk;                               // local layout: number of route blocks

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef MOE_WAIT_STATS
  const long long _k0 = clock64();
#endif
  pdl_launch_dependents();
  if (threadIdx.x == 0) MOE_TL(3 + a.stage, 0);
  const int total_tiles = a.num_blocks * a.n_tiles;
  const int kblocks = a.K / kTileK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int j = 0; j < C::kASlots; ++j) {
      mbar_init(&a_full[j], C::kConvWarps);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // Decode sizes: the route layout is derived from topk_ids before the
  // dependency wait (see local_block_layout), so the producer loads its first
  // weight tiles while the previous kernel still runs.
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

  auto stage_ptr = [&](int s) { return smem + s * C::kStageBytes; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // A second cursor runs kPrefetch weight tiles ahead and prefetches them
    // (contiguous 8 KB blocks) and their scale atoms into L2. With the local
    // layout the weight half of the first ring stages (packed tile and scale
    // atom) is loaded before the dependency wait and the activation half
    // after it.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int kPrefetch = a.prefetch;   // per call; 8 by default
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_mask = 0, armed_par = 0;   // stages armed, parity of their last arming
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
        int pf_kb = seq_kb0(pf);
        auto pf_skip = [&]() {
          if (++pf_kb == seq_kb1(pf, kblocks)) {
            seq_next(pf, a, total_tiles, P, BN);
            if (pf.valid) pf_kb = seq_kb0(pf);
          }
        };
        auto pf_step = [&]() {
          if (!pf.valid) return;
          const int64_t tile =
              (static_cast<int64_t>(expert_of(pf)) * a.n_tiles + pf.n_tile) * kblocks + pf_kb;
          // with the unit's weight scale atoms (512 B per k-block, contiguous)
          if (pf_kb == seq_kb0(pf))
            bulk_prefetch_l2(a.sfa + tile * 512,
                             static_cast<uint32_t>(seq_kb1(pf, kblocks) - pf_kb) * 512);
          bulk_prefetch_l2(a.w + tile * C::kRawBytes, C::kRawBytes);
          pf_skip();
        };
        int kb = 0, kb_end = 0;
        int64_t tile0 = 0;
        auto set_tile = [&]() {
          tile0 = (static_cast<int64_t>(expert_of(cur)) * a.n_tiles + cur.n_tile) * kblocks;
          kb = seq_kb0(cur);
          kb_end = seq_kb1(cur, kblocks);
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
          uint8_t* sb = stage_ptr(stage);
          tma_load_2d(sb + C::kBBytes, &tmW, &full_bar[stage], 0,
                      static_cast<int32_t>((tile0 + kb) * kTileN), pol_w);
          bulk_load(sb + C::kBBytes + C::kRawBytes, a.sfa + (tile0 + kb) * 512, 512,
                    &full_bar[stage], pol_w);
        };
        auto load_x = [&](int st, int kbx, int m_blk) {
          uint8_t* sb = stage_ptr(st);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sb + h * C::kBAtomBytes, &tmX, &full_bar[st], kbx * kTileK + h * kAtomK,
                        m_blk * BN, pol_x);
        };
        auto advance = [&](bool prefetch) {
          if (prefetch) pf_step();
          else if (pf.valid) pf_skip();
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
          if (++kb == kb_end) {
            seq_next(cur, a, total_tiles, P, BN);
            if (cur.valid) set_tile();
          }
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
          int npre = 0;
          int pre_kb[C::kStages], pre_m[C::kStages];
          while (cur.valid && npre < C::kStages) {
            arm();
            load_w();
            pre_kb[npre] = kb;
            pre_m[npre] = cur.m_blk;
            ++npre;
            advance(false);   // these k-blocks are being loaded, not prefetched
          }
          for (int i = 0; i < kPrefetch; ++i) pf_step();
          pdl_wait_prior();
          if (threadIdx.x == 0) MOE_TL(3 + a.stage, 1);
          for (int i = 0; i < npre; ++i) load_x(i, pre_kb[i], pre_m[i]);
        }
        while (cur.valid && !abort_flag) {
          bool ok;
          { WS_T0(); ok = mbar_wait(&empty_bar[stage], phase ^ 1, a.status); WS_ADD(0); }
          if (!ok) { abort_flag = 1; break; }
          arm();
          load_w();
          load_x(stage, kb, cur.m_blk);
          advance(true);
        }
        if constexpr (kLocal) {
          // the layout derived from topk_ids must be the sort's
          if (*a.num_padded != P && a.status) atomicOr(a.status, kDevBadExpert);
        }
      };
      if (a.local)
        produce(Seq16R{}, [&](const Seq16R& q) { return static_cast<int>(s_blk_expert[q.m_blk]); },
                std::true_type{});
      else
        produce(Seq16{}, [](const Seq16& q) { return q.e; }, std::false_type{});
      // Copies still in flight into shared memory must land before the CTA
      // exits: normally every armed stage was consumed, so these return at
      // once; after an abort they wait (bounded) for the TMA.
      for (int s = 0; s < C::kStages; ++s)
        if ((armed_mask >> s) & 1u) mbar_wait(&full_bar[s], (armed_par >> s) & 1u, a.status);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    pdl_wait_prior();
    const int P = a.local ? s_nblk * BN : *a.num_padded;
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t slot_phase = 0;
      int local = 0;
#ifdef MOE_TIMELINE
      int tl_mma = 1;
#endif
      constexpr uint32_t idesc = idesc_dense(1, 1, kTileN, BN);
      const uint64_t b_desc0 = smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
      Seq16R seq;
      for (seq_init(seq, a, total_tiles, P, BN, kblocks); seq.valid && !abort_flag;
           seq_next(seq, a, total_tiles, P, BN)) {
        const int ab = local % C::kAccBufs;
        const uint32_t acc_phase = (local / C::kAccBufs) & 1;
        ++local;
        bool ok0;
        { WS_T0(); ok0 = mbar_wait(&acc_empty[ab], acc_phase ^ 1, a.status); WS_ADD(3); }
        if (!ok0) { abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + C::kAccCol0 + ab * BN;
        const int kb_begin = seq_kb0(seq), kb_end = seq_kb1(seq, kblocks);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          bool ok1, ok2;
          { WS_T0(); ok1 = mbar_wait(&full_bar[stage], phase, a.status); WS_ADD(1); }
          { WS_T0(); ok2 = ok1 && mbar_wait(&a_full[slot], slot_phase, a.status); WS_ADD(2); }
          if (!ok2) { abort_flag = 1; break; }
#ifdef MOE_TIMELINE
          if (tl_mma) { MOE_TL(3 + a.stage, 3); tl_mma = 0; }
#endif
          tc_fence_after();
          const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage) * (C::kStageBytes >> 4);
          const uint32_t a_tmem = tmem + slot * kACols;
#pragma unroll
          for (int kk = 0; kk < kTileK / kMmaK; ++kk) {
            // B: atom h of the stage, then 32 bytes (2 descriptor units) per MMA;
            // A: 8 TMEM columns (16 BF16) per MMA
            const int h = kk / (kAtomK / kMmaK), off = (kk % (kAtomK / kMmaK)) * 2;
            mma_f16_tmem_a(d_tmem, a_tmem + kk * (kMmaK / 2),
                           bd + h * (C::kBAtomBytes >> 4) + off, idesc, kb > kb_begin || kk != 0);
          }
          tc_commit(&empty_bar[stage]);         // frees the smem stage and the TMEM slot
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
          if (++slot == C::kASlots) { slot = 0; slot_phase ^= 1; }
        }
        tc_commit(&acc_full[ab]);
      }
      MOE_TL(3 + a.stage, 4);
      tc_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, a.status);
    }
  } else if (warp >= 6) {
    // ---------------------------------------------------------- converters
    pdl_wait_prior();
    const int P = a.local ? s_nblk * BN : *a.num_padded;
    constexpr int kHalves = C::kConvWarps == 8 ? 1 : 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                      // weight row = TMEM lane
    const int h0 = C::kConvWarps == 8 ? (warp - 6) >> 2 : 0;
    const int swz = (r >> 1) & 3;                        // 64-byte swizzle of row r
    const int sf_off = sf_atom_off(r, 0);                // its 4 scale bytes
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;                 // TMEM slot of this k-block
    int lag_stage = 0;            // stage of k-block j - kASlots, whose MMA frees the slot
    uint32_t lag_phase = 0;
    int done = 0;                 // k-blocks converted so far
    Seq16R seq;
    for (seq_init(seq, a, total_tiles, P, BN, kblocks); seq.valid;
         seq_next(seq, a, total_tiles, P, BN)) {
      bool stop = false;
      for (int kb = seq_kb0(seq); kb < seq_kb1(seq, kblocks); ++kb) {
        bool okc1 = !abort_flag, okc2;
#ifdef MOE_WAIT_STATS
        const bool rep = threadIdx.x == 192;
#endif
        { WS_T0(); okc1 = okc1 && mbar_wait(&full_bar[stage], phase, a.status);
#ifdef MOE_WAIT_STATS
          if (rep) WS_ADD(4);
#endif
        }
        okc2 = okc1;
        if constexpr (C::kStages > C::kASlots) {
          // the slot is free once the MMA of k-block j - kASlots committed;
          // with equal rings the landed stage implies it (the producer
          // reloaded the stage only after that commit)
          if (okc2 && done >= C::kASlots) {
            WS_T0();
            okc2 = mbar_wait(&empty_bar[lag_stage], lag_phase, a.status);
#ifdef MOE_WAIT_STATS
            if (rep) WS_ADD(5);
#endif
            if (++lag_stage == C::kStages) { lag_stage = 0; lag_phase ^= 1; }
          }
        }
#ifdef MOE_WAIT_STATS
        const long long _cb0 = clock64();
#endif
        if (!okc2) {
          abort_flag = 1; stop = true; break;
        }
        tc_fence_after();
        const uint8_t* raw = stage_ptr(stage) + C::kBBytes + r * 64;
        const uint32_t sfw =
            *reinterpret_cast<const uint32_t*>(stage_ptr(stage) + C::kBBytes + C::kRawBytes + sf_off);
        // a scale byte above 128 in one of the warp's rows (never for real
        // weights): the warp converts this k-block with a second multiplication
        const bool big = __any_sync(0xffffffffu, a16_big_scales(sfw) != 0u);
        const uint32_t tsc = sfw + 0x7E7E7E7Eu;           // s + 126 per byte when !big
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          const int h = h0 + hh;                           // 64-element half of the stage
          uint32_t out[32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {                 // 32 elements = one scale block
            const int c = 2 * h + cc;
            const uint4 v = *reinterpret_cast<const uint4*>(raw + ((c ^ swz) << 4));
            const uint32_t sb = (sfw >> (8 * c)) & 0xFFu;
            uint32_t pairs[16];
            a16_dequant_block(v, big ? a16_first_pair(sb) : a16_scale_pair(tsc, c), pairs);
            if (big) {
              const uint32_t sc2 = a16_big_pair(sb);
#pragma unroll
              for (int i = 0; i < 16; ++i) pairs[i] = a16_bf16x2_mul(pairs[i], sc2);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) out[cc * 16 + i] = pairs[i];
          }
          tmem_st_32x32b_x32(t_row + slot * kACols + h * 32, out);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[slot]);
#ifdef MOE_WAIT_STATS
        if (rep)
          atomicAdd(reinterpret_cast<unsigned long long*>(&g_ws16[blockIdx.x & 511][a.stage - 1][6]),
                    static_cast<unsigned long long>(clock64() - _cb0));
#endif
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        if (++slot == C::kASlots) slot = 0;
        ++done;
      }
      if (stop) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait_prior();
    const int P = a.local ? s_nblk * BN : *a.num_padded;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int et = threadIdx.x - 64;
    const int R = a.M * a.topk;
    int local = 0;
    Seq16R seq;
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
      bool oke = !abort_flag;
      { WS_T0(); oke = oke && mbar_wait(&acc_full[ab], acc_phase, a.status);
#ifdef MOE_WAIT_STATS
        if (threadIdx.x == 64) WS_ADD(7);
#endif
      }
      if (!oke) { abort_flag = 1; break; }
      tc_fence_after();
      const uint32_t d_tmem =
          tmem + C::kAccCol0 + ab * BN + (static_cast<uint32_t>(quad * 32) << 16);
      const int64_t p_base = static_cast<int64_t>(m_blk) * BN;
      constexpr int kChunk = BN < 32 ? BN : 32;
      auto load_acc = [&](int c0, float (&v)[32]) {
        uint32_t r32[32];
        if constexpr (kChunk == 32) {
          tmem_ld_32x32b_x32(d_tmem + c0, r32);
        } else {
          uint32_t r16[16];
          tmem_ld_32x32b_x16(d_tmem + c0, r16);
#pragma unroll
          for (int i = 0; i < 16; ++i) r32[i] = r16[i];
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kChunk; ++i) v[i] = __uint_as_float(r32[i]);
      };
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
            load_acc(c0, v);
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
      // from the split slot for the last part of a split stage-1 tile); two
      // loops keep the TMEM path free of the slot pointer (with it in one
      // loop the a8w4 split kernel's stage 2 ran 2x slower).
      auto finish = [&](const int c0, float (&v)[32]) {
        if (a.stage == 1) {
          // gate/up pairs in adjacent lanes; even lanes take columns [0, half)
          constexpr int half = kChunk / 2;
          const bool odd = lane & 1;
          const int j_local = row >> 1;
          named_bar_sync(1, 128);
#pragma unroll
          for (int k = 0; k < half; ++k) {
            const float send = odd ? v[k] : v[k + half];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float gate = odd ? recv : v[k];
            const float up = odd ? v[k + half] : recv;
            epi[(k + (odd ? half : 0)) * 68 + j_local] = __fdividef(gate, 1.0f + __expf(-gate)) * up;
          }
          named_bar_sync(1, 128);
          const int item = et >> 1, hf = et & 1;
          const int col = item >> 1, blk = item & 1;
          if (col < kChunk) {
            const int64_t p = p_base + c0 + col;
            const bool pad = s_tok[c0 + col] < 0;
            const float4* src =
                reinterpret_cast<const float4*>(epi + col * 68 + blk * 32 + hf * 16);
            uint32_t o[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 f = src[q];
              __nv_bfloat162 h0 = __floats2bfloat162_rn(f.x, f.y);
              __nv_bfloat162 h1 = __floats2bfloat162_rn(f.z, f.w);
              o[2 * q] = pad ? 0u : *reinterpret_cast<uint32_t*>(&h0);
              o[2 * q + 1] = pad ? 0u : *reinterpret_cast<uint32_t*>(&h1);
            }
            const int jcol = n_tile * 64 + blk * 32 + hf * 16;
            uint4* dst = reinterpret_cast<uint4*>(a.inter + p * a.Ip + jcol);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        } else if constexpr (BN >= 64) {
          // stage 2, large tiles: the chunk's weighted values go through
          // shared memory route-major (8 routes x 128 features per pass, two
          // alternating buffers, one barrier per pass), and each warp then adds
          // whole 512-byte token-row segments with 16-byte vector reductions
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
          load_acc(c0, v);
          finish(c0, v);
        }
      }
      if (!part) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
      }
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
#ifdef MOE_WAIT_STATS
  if (threadIdx.x == 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(&g_ws16[blockIdx.x & 511][a.stage - 1][8]),
              static_cast<unsigned long long>(clock64() - _k0));
#endif
  if (threadIdx.x == 0) {
    MOE_TL(3 + a.stage, 7);
  }
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
               uint64_t rows, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle sw) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess || q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t plan_bn(const Bf16Args& a, int split, int num_sms, GemmPlan* plan) {
  using C = Cfg16<BN>;
  static_assert(sizeof(Bf16Args) <= sizeof(plan->args), "argument block");
  const int tiles = a.num_blocks * a.n_tiles;
  const int slots = num_sms * C::kCtasPerSm;
  // The split-walk kernel as for a8w4: at route blocks <= 32 unless the
  // call asks for whole tiles (split = 2). Stage 1 needs the split slots.
  const void* fn = reinterpret_cast<const void*>(&moe_gemm_bf16w4_kernel<BN, false>);
  if constexpr (BN <= 32) {
    if (split != 2 && (a.stage == 2 || a.split_part))
      fn = reinterpret_cast<const void*>(&moe_gemm_bf16w4_kernel<BN, true>);
  }
  cudaError_t err = ensure_smem_attr(fn, C::kSmem);
  if (err != cudaSuccess) return err;
  plan->kernel = fn;
  const bool split_kernel = fn != reinterpret_cast<const void*>(&moe_gemm_bf16w4_kernel<BN, false>);
  plan->grid = split_kernel || tiles > slots ? slots : tiles;
  plan->threads = C::kThreads;
  plan->smem = C::kSmem;
  memcpy(plan->args, &a, sizeof(a));
  return cudaSuccess;
}

}  // namespace

cudaError_t prepare_gemm_bf16w4(int stage, const GemmArgs& g, GemmPlan* plan) {
  Bf16Args a{};
  a.stage = stage;
  a.M = g.M; a.topk = g.topk; a.H = g.H; a.Ip = g.Ip; a.E = g.E;
  a.N = stage == 1 ? 2 * g.Ip : g.H;
  a.K = stage == 1 ? g.H : g.Ip;
  a.n_tiles = a.N / kTileN;
  a.num_blocks = static_cast<int>(g.p_max / g.bm);
  a.n_group_log2 = stage == 1 ? 0 : stage2_n_group_log2(g.M, g.p_max * g.Ip * 2, a.n_tiles);
  a.local = (g.topk_ids || g.gate.logits) &&
            static_cast<int64_t>(g.M) * g.topk <= kLocalMaxRoutes &&
            a.num_blocks <= kLocalMaxBlocks ? 1 : 0;
  a.topk_ids = g.topk_ids;
  a.gate = g.gate;
  a.sorted_route = g.sorted_route; a.sorted_w = g.sorted_w; a.block_expert = g.block_expert;
  a.num_padded = g.num_padded;
  a.sfa = stage == 1 ? g.w1s : g.w2s;
  a.w = stage == 1 ? g.w1 : g.w2;
  a.inter = static_cast<__nv_bfloat16*>(g.inter);
  a.acc = g.acc;
  a.prefetch = stage == 1 ? (g.prefetch1 > 0 ? g.prefetch1 : 8)
                         : (g.prefetch2 > 0 ? g.prefetch2 : 8);
  a.status = g.status;
  a.split_part = g.split_part;
  a.split_cnt = g.split_cnt;
  plan->grid = 0;
  if (a.num_blocks == 0) return cudaSuccess;
  const void* xb = stage == 1 ? g.act : g.inter;
  CUtensorMap* tw = reinterpret_cast<CUtensorMap*>(plan->tmap_a);
  CUtensorMap* tx = reinterpret_cast<CUtensorMap*>(plan->tmap_b);
  // packed weight tiles as rows of 64 bytes, one 128-row box per tile, 64-byte swizzle
  const uint64_t w_rows = static_cast<uint64_t>(g.E) * a.n_tiles * (a.K / kTileK) * kTileN;
  if (!encode_2d(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, 64, w_rows, 64, 64, kTileN,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (!encode_2d(tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, a.K, static_cast<uint64_t>(g.p_max),
                 static_cast<uint64_t>(a.K) * 2, kAtomK, g.bm, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  switch (g.bm) {
    case 16: return plan_bn<16>(a, g.split, sms, plan);
    case 32: return plan_bn<32>(a, g.split, sms, plan);
    case 64: return plan_bn<64>(a, g.split, sms, plan);
    case 128: return plan_bn<128>(a, g.split, sms, plan);
    case 256: return plan_bn<256>(a, g.split, sms, plan);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe

#ifdef MOE_WAIT_STATS
extern "C" void moe_debug_wait_stats16(long long* host_out, int reset) {
  cudaMemcpyFromSymbol(host_out, moe::g_ws16, sizeof(moe::g_ws16));
  if (reset) {
    static long long zeros[512][2][16] = {};
    cudaMemcpyToSymbol(moe::g_ws16, zeros, sizeof(zeros));
  }
}
#endif
