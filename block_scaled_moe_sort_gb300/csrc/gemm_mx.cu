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
//   A  E2M1, expanded by TMA (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B) to 16-byte
//      units holding 16 codes in their low 8 bytes, i.e. one byte slot per
//      element as kind::mxf8f6f4 expects for 4-bit operands;
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
#include <cuda.h>
#include <cudaTypedefs.h>
#include "common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

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
  const int32_t* sorted_route;
  const float* sorted_w;
  const int32_t* block_expert;
  const int32_t* num_padded;
  const uint8_t* sfa;    // weight scale atoms [E][N/128][K/128][512]
  const uint8_t* sfb;    // route scale atoms [blocks][K/128][na][512]
  uint8_t* inter;        // stage 1 out: E4M3 [p_max, Ip]
  uint8_t* inter_sf;     // stage 1 out: atoms [blocks][Ip/128][na][512]
  float* acc;            // stage 2 out: [M, H]
  int32_t* status;
};

template <int BN>
struct Cfg {
  static constexpr int kNa = (BN + 127) / 128;                 // scale atoms per B stage
  static constexpr int kABytes = kTileN * kTileK;              // 16 KB (expanded FP4)
  static constexpr int kBBytes = BN * kTileK;
  static constexpr int kSfBytes = 512 * (1 + kNa);
  static constexpr int kStageBytes = (kABytes + kBBytes + kSfBytes + 1023) / 1024 * 1024;
  static constexpr int kStages = BN <= 32 ? 8 : (BN <= 64 ? 7 : (BN <= 128 ? 5 : 4));
  static constexpr int kAccBufs = BN <= 128 ? 2 : 1;
  static constexpr int kSfCols = 4 * (1 + kNa);                // TMEM columns per stage
  static constexpr int kColsNeeded = kAccBufs * BN + kStages * kSfCols;
  static constexpr int kTmemCols = kColsNeeded <= 32 ? 32 : kColsNeeded <= 64 ? 64
                                   : kColsNeeded <= 128 ? 128 : kColsNeeded <= 256 ? 256 : 512;
  static constexpr int kEpiFloats = 32 * (64 + 4);             // stage-1 transpose tile
  static constexpr int kSmem = 1024 /*align slack*/ + kStages * kStageBytes + kEpiFloats * 4 + 256;
  // TMA transaction bytes of one stage: FP4 A counts packed bytes
  static constexpr uint32_t kTxBytes = kTileN * kTileK / 2 + kBBytes + kSfBytes;
  static_assert(kColsNeeded <= 512, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "smem budget");
};

__device__ __forceinline__ void tile_coords(int t, const MxArgs& a, int& m_blk, int& n_tile) {
  if (a.stage == 1) {  // route-block major: the n-tiles of a block share its activations
    m_blk = t / a.n_tiles;
    n_tile = t % a.n_tiles;
  } else {             // feature-tile major: the FP32 reductions of a tile stay in L2
    n_tile = t / a.num_blocks;
    m_blk = t % a.num_blocks;
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const MxArgs a) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* epi = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  __shared__ uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  __shared__ uint64_t acc_full[C::kAccBufs], acc_empty[C::kAccBufs];
  __shared__ uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = *a.num_padded;
  const int total_tiles = a.num_blocks * a.n_tiles;
  const int kblocks = a.K / kTileK;

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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sf_col0 = C::kAccBufs * BN;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();   // weights: streamed once
      const uint64_t pol_x = policy_evict_last();    // routes: reused across n-tiles
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total_tiles && !abort_flag; t += gridDim.x) {
        int m_blk, n_tile;
        tile_coords(t, a, m_blk, n_tile);
        if (m_blk * BN >= P) continue;
        const int e = __ldg(a.block_expert + m_blk);
        if (e < 0 || e >= a.E) continue;
        const int row_a = e * a.N + n_tile * kTileN;
        const uint8_t* sfa = a.sfa + ((static_cast<int64_t>(e) * a.n_tiles + n_tile) * kblocks) * 512;
        const uint8_t* sfb = a.sfb + static_cast<int64_t>(m_blk) * kblocks * C::kNa * 512;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, a.status)) { abort_flag = 1; break; }
          uint8_t* sbase = stages + stage * C::kStageBytes;
          mbar_arrive_expect_tx(&full_bar[stage], C::kTxBytes);
          tma_load_2d(sbase, &tmA, &full_bar[stage], kb * kTileK, row_a, pol_w);
          tma_load_2d(sbase + C::kABytes, &tmB, &full_bar[stage], kb * kTileK, m_blk * BN, pol_x);
          bulk_load(sbase + C::kABytes + C::kBBytes, sfa + kb * 512, 512, &full_bar[stage], pol_w);
          bulk_load(sbase + C::kABytes + C::kBBytes + 512, sfb + kb * C::kNa * 512,
                    512 * C::kNa, &full_bar[stage], pol_x);
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int t = blockIdx.x; t < total_tiles && !abort_flag; t += gridDim.x) {
        int m_blk, n_tile;
        tile_coords(t, a, m_blk, n_tile);
        if (m_blk * BN >= P) continue;
        const int e = __ldg(a.block_expert + m_blk);
        if (e < 0 || e >= a.E) continue;
        const int ab = local % C::kAccBufs;
        const uint32_t acc_phase = (local / C::kAccBufs) & 1;
        ++local;
        if (!mbar_wait(&acc_empty[ab], acc_phase ^ 1, a.status)) { abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + ab * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, a.status)) { abort_flag = 1; break; }
          tc_fence_after();
          uint8_t* sbase = stages + stage * C::kStageBytes;
          const uint32_t a_addr = smem_u32(sbase);
          const uint32_t b_addr = smem_u32(sbase + C::kABytes);
          const uint32_t sf_addr = smem_u32(sbase + C::kABytes + C::kBBytes);
          const uint32_t sfa_t = tmem + sf_col0 + stage * C::kSfCols;
          const uint32_t sfb_t = sfa_t + 4;
          tmem_cp_32x128b_warpx4(sfa_t, smem_desc(sf_addr, 0, 128, kSwizzleNone));
#pragma unroll
          for (int j = 0; j < C::kNa; ++j)
            tmem_cp_32x128b_warpx4(sfb_t + 4 * j,
                                   smem_desc(sf_addr + 512 * (1 + j), 0, 128, kSwizzleNone));
#pragma unroll
          for (int kk = 0; kk < kTileK / kMmaK; ++kk) {
            const uint64_t ad = smem_desc(a_addr + kk * kMmaK, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(b_addr + kk * kMmaK, 16, 1024, kSwizzle128B);
            mma_mxf8f6f4(d_tmem, ad, bd, idesc_mx(5, 0, kTileN, BN, kk, kk), sfa_t, sfb_t,
                         (kb | kk) != 0);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
        tc_commit(&acc_full[ab]);
      }
      // every MMA issued by this thread has finished before TMEM is released
      tc_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, a.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;               // TMEM lane quadrant
    const int row = quad * 32 + lane;        // weight row within the tile
    const int et = threadIdx.x - 64;         // 0..127
    const int R = a.M * a.topk;
    int local = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      int m_blk, n_tile;
      tile_coords(t, a, m_blk, n_tile);
      if (m_blk * BN >= P) continue;
      const int e = __ldg(a.block_expert + m_blk);
      if (e < 0 || e >= a.E) continue;
      const int ab = local % C::kAccBufs;
      const uint32_t acc_phase = (local / C::kAccBufs) & 1;
      ++local;
      if (abort_flag || !mbar_wait(&acc_full[ab], acc_phase, a.status)) { abort_flag = 1; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem + ab * BN + (static_cast<uint32_t>(quad * 32) << 16);
      const int64_t p_base = static_cast<int64_t>(m_blk) * BN;
      constexpr int kChunk = BN < 32 ? BN : 32;
      for (int c0 = 0; c0 < BN; c0 += kChunk) {
        float v[32];
        {
          uint32_t r[32];
          if constexpr (kChunk == 32) {
            tmem_ld_32x32b_x32(d_tmem + c0, r);
          } else {
            uint32_t r16[16];
            tmem_ld_32x32b_x16(d_tmem + c0, r16);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = r16[i];
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < kChunk; ++i) v[i] = __uint_as_float(r[i]);
        }
        if (a.stage == 1) {
          // gate (even row) / up (odd row) pairs sit in adjacent lanes
          const int j_local = row >> 1;       // 0..63
          named_bar_sync(1, 128);             // previous chunk's readers are done
#pragma unroll
          for (int i = 0; i < kChunk; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, v[i], 1);
            if ((lane & 1) == 0) epi[i * 68 + j_local] = silu_mul(v[i], other);
          }
          named_bar_sync(1, 128);
          // 2 threads per (route column, 32-block): each quantises 16 values
          const int item = et >> 1, half = et & 1;     // 64 items
          const int col = item >> 1, blk = item & 1;   // column in chunk, 32-block in tile
          if (col < kChunk) {
            const int64_t p = p_base + c0 + col;
            const bool pad = __ldg(a.sorted_route + p) >= R;
            float x[16];
            const float4* src = reinterpret_cast<const float4*>(epi + col * 68 + blk * 32 + half * 16);
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
            const int jcol = n_tile * 64 + blk * 32 + half * 16;   // intermediate column
            *reinterpret_cast<uint4*>(a.inter + p * a.Ip + jcol) =
                make_uint4(codes[0], codes[1], codes[2], codes[3]);
            if (half == 0) {
              const int ib = jcol / 32;                          // 32-block index along Ip
              const int rr = static_cast<int>(p % BN);
              const int64_t atom = (static_cast<int64_t>(m_blk) * (a.Ip / 128) + ib / 4) * C::kNa + rr / 128;
              a.inter_sf[atom * 512 + sf_atom_off(rr & 127, ib & 3)] = static_cast<uint8_t>(sb);
            }
          }
        } else {
          // route info of this chunk's columns, one per lane, broadcast by shuffle
          int tok = -1;
          float wgt = 0.f;
          if (lane < kChunk) {
            const int64_t p = p_base + c0 + lane;
            const int r = __ldg(a.sorted_route + p);
            if (r < R) { tok = r / a.topk; wgt = __ldg(a.sorted_w + p); }
          }
          const int n = n_tile * kTileN + row;
#pragma unroll
          for (int i = 0; i < kChunk; ++i) {
            const int ti = __shfl_sync(0xffffffffu, tok, i);
            const float wi = __shfl_sync(0xffffffffu, wgt, i);
            if (ti >= 0) atomicAdd(a.acc + static_cast<int64_t>(ti) * a.H + n, wi * v[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

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
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const MxArgs& a,
                      int num_sms, cudaStream_t s) {
  using C = Cfg<BN>;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(&moe_gemm_mx_kernel<BN>),
                                     C::kSmem);
  if (err != cudaSuccess) return err;
  const int tiles = a.num_blocks * a.n_tiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  moe_gemm_mx_kernel<BN><<<grid, kThreads, C::kSmem, s>>>(ta, tb, a);
  return cudaGetLastError();
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

}  // namespace

cudaError_t launch_gemm_mx(int stage, const GemmArgs& g, cudaStream_t s) {
  MxArgs a{};
  a.stage = stage;
  a.M = g.M; a.topk = g.topk; a.H = g.H; a.Ip = g.Ip; a.E = g.E;
  a.N = stage == 1 ? 2 * g.Ip : g.H;
  a.K = stage == 1 ? g.H : g.Ip;
  a.n_tiles = a.N / kTileN;
  a.num_blocks = static_cast<int>(g.p_max / g.bm);
  a.sorted_route = g.sorted_route; a.sorted_w = g.sorted_w; a.block_expert = g.block_expert;
  a.num_padded = g.num_padded;
  a.sfa = stage == 1 ? g.w1s : g.w2s;
  a.sfb = stage == 1 ? g.act_sf : g.inter_sf;
  a.inter = static_cast<uint8_t*>(g.inter);
  a.inter_sf = g.inter_sf;
  a.acc = g.acc;
  a.status = g.status;
  if (a.num_blocks == 0) return cudaSuccess;

  CUtensorMap ta, tb;
  const uint8_t* w = stage == 1 ? g.w1 : g.w2;
  const void* xb = stage == 1 ? g.act : g.inter;
  if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, a.K,
                 static_cast<uint64_t>(a.E) * a.N, a.K / 2, 128, kTileN))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, xb, a.K, static_cast<uint64_t>(g.p_max), a.K,
                 128, g.bm))
    return cudaErrorInvalidValue;
  const int sms = sm_count();
  switch (g.bm) {
    case 16: return launch_bn<16>(ta, tb, a, sms, s);
    case 32: return launch_bn<32>(ta, tb, a, sms, s);
    case 64: return launch_bn<64>(ta, tb, a, sms, s);
    case 128: return launch_bn<128>(ta, tb, a, sms, s);
    case 256: return launch_bn<256>(ta, tb, a, sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
