/*
 * moe_mx.h - C ABI of the GB300 (sm_103a) block-scaled fused MoE layer.
 *
 * One call of the layer (a8w4 variant) does, on one CUDA stream:
 *   sort    token-expert routes grouped by expert, each group padded to
 *           block_m ("the sorter": AITER #5609 "Add DeepSeek V4.1 Flash TP4
 *           gfx950 MoE tuning", Performance on the measured runtime; sorting
 *           is part of the timed call in AITER #5904 "Add tuned a8w4
 *           fused-MoE configs for DeepSeek V4.1-Flash (TP4 + EP, gfx950)",
 *           Fused-MoE kernel expert-parallel benchmark)
 *   quant   BF16 tokens -> FP8 E4M3 + one E8M0 scale per 1x32 along K
 *           (AITER #5609, Configuration: FP8 activations, per-1x32 scaling)
 *   stage 1 grouped GEMM against interleaved gate/up MXFP4 expert rows,
 *           SiLU(gate)*up with no routing-weight multiply, requantised to
 *           per-1x32 FP8 (AITER #5609, Configuration; "the intermediate
 *           quantization", AITER #5904, Fused-MoE kernel benchmark)
 *   stage 2 grouped down-projection GEMM; the routing-weighted sum over a
 *           token's routes is reduced into a BF16 output (AITER #5609,
 *           Configuration: BF16 output)
 * The a16w4 variant keeps BF16 activations and a BF16 intermediate
 * (AITER #6286 "Retune gfx942 a16w4 DSv4.1 tiles for Triton 3.8", reviewer
 * reply: moe_gemm_a16w4, w1 with apply_swiglu=True, w2 separate, bf16,
 * MXFP4).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated; the caller owns all memory.
 *    The library never allocates, frees or synchronises, and never reads
 *    device data on the host, so every call can be captured in a CUDA graph
 *    (all launch shapes depend only on the integer arguments).
 *  - Inputs are const and never written.
 *  - Argument errors return synchronously before any launch, leaving every
 *    buffer untouched. Launch failures return MOE_ERR_CUDA (from
 *    cudaGetLastError). Device-side faults the kernels detect themselves (a
 *    pipeline wait that timed out) set bits in the workspace status word, see
 *    moe_ws_layout_t.status_off.
 *  - Layouts are row-major. E2M1 codes are packed two per byte: element k in
 *    byte k/2, low nibble = even k. E8M0 scale bytes hold 2^(b-127), one per
 *    32 consecutive elements along K. In w1 row 2j is gate_j and row 2j+1 is
 *    up_j. Device pointers must be 256-byte aligned; the stream is a
 *    cudaStream_t (0 = legacy default stream).
 */
#ifndef MOE_MX_H
#define MOE_MX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* == cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size */
  MOE_ERR_UNSUPPORTED = 2,  /* a shape outside what the kernels implement */
  MOE_ERR_WORKSPACE = 3,    /* workspace smaller than the *_workspace_bytes size */
  MOE_ERR_ALIGNMENT = 4,    /* a pointer not 256-byte aligned */
  MOE_ERR_CUDA = 5,         /* a CUDA runtime/driver call or a launch failed */
  MOE_ERR_TIMEOUT = 6,      /* reported by moe_decode_device_status */
  MOE_ERR_DEVICE_CHECK = 7  /* reported by moe_decode_device_status: a route block
                               reached a GEMM with an expert id outside [0, E) */
} moe_status_t;

/* Static text for a status code (never NULL). */
const char* moe_status_string(moe_status_t s);

/* ------------------------------------------------------------------ sort
 * moe_sort: stable counting sort of the M*topk routes by expert id.
 * Route r = t*topk + j (token t, slot j) goes to expert topk_ids[r]; routes
 * whose id is outside [0, E) are dropped (expert-parallel shard). Within an
 * expert routes keep ascending r. Each non-empty expert's segment is padded
 * to a multiple of block_m; empty experts take no block.
 *
 * Outputs (device, caller-allocated, sizes from moe_sort_max_padded):
 *   sorted_route [P_max] int32  route r per sorted position; pad = M*topk
 *   sorted_w     [P_max] float  topk_weights[r]; pad = 0
 *   block_expert [P_max/block_m] int32  expert of each block_m block; -1
 *                for blocks at or beyond num_padded
 *   expert_off   [E+1]   int32  padded segment starts, expert_off[E] = P
 *   num_padded   [1]     int32  P = sum_e ceil(cnt_e/block_m)*block_m
 *   route_pos    [M*topk] int32 sorted position of r, -1 if dropped
 *                (may be NULL)
 * ws/ws_bytes: scratch of at least moe_sort_workspace_bytes (may be NULL when
 * that is 0); MOE_ERR_WORKSPACE if too small.
 * Positions in [P, P_max) are filled with the pad sentinel. When P_max is 0
 * (M == 0) the three P_max-sized outputs may be NULL.
 * Limits: 1 <= E <= 512, 1 <= topk <= 16, block_m in {16,32,64,128,256},
 * M*topk <= 2^24. M == 0 is allowed (writes the empty result).
 */
int64_t moe_sort_max_padded(int M, int topk, int E, int block_m);
/* Scratch the sort needs (device, caller-allocated): 0 up to 8192 routes,
 * else 4*E bytes per 8192 routes (per-CTA expert histograms). */
size_t moe_sort_workspace_bytes(int M, int topk, int E, int block_m);
moe_status_t moe_sort(const int32_t* topk_ids, const float* topk_weights, int M, int topk,
                      int E, int block_m, int32_t* sorted_route, float* sorted_w,
                      int32_t* block_expert, int32_t* expert_off, int32_t* num_padded,
                      int32_t* route_pos, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------ gating
 * moe_router_topk: router logits -> topk_ids / topk_weights for moe_sort and
 * the fused calls (the gating the pages time together with the layer, AITER
 * #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the
 * measured runtime). Per token t:
 *   - the topk experts with the largest logits[t, e]; equal logits are taken
 *     in ascending expert order; columns are in that order (descending
 *     logit, then ascending expert);
 *   - weight of a pick = softmax of the picks' logits (FP32 arithmetic);
 *   - if shared_id >= 0, n_shared more columns hold shared_id, shared_id + 1,
 *     ..., each with weight 1.0 (the 385-expert top-7 layout: one shared
 *     expert, id E; a shared expert whose intermediate is split into
 *     n_shared pieces of the routed experts' size takes n_shared ids).
 * logits: float32 [M, E], row stride ld >= E elements, finite values.
 * topk_ids int32 / topk_weights float32: [M, topk (+ n_shared)],
 *   caller-allocated device memory, fully written.
 * Errors (before any launch): MOE_ERR_INVALID_ARG for M < 0, E < 1, ld < E,
 * topk outside [1, E], shared_id >= 0 with shared_id < E (a shared expert
 * comes after the E routed experts), n_shared < 1 or shared_id + n_shared >
 * 512, or a NULL pointer with M > 0; MOE_ERR_UNSUPPORTED for E > 512 or more
 * than 16 output columns; MOE_ERR_ALIGNMENT for pointers not 256-byte
 * aligned. n_shared is ignored when shared_id < 0. M == 0 launches nothing.
 */
moe_status_t moe_router_topk(const float* logits, int M, int E, int ld, int topk, int shared_id,
                             int n_shared, int32_t* topk_ids, float* topk_weights,
                             moe_stream_t stream);

/* -------------------------------------------------------- activation quant
 * moe_quant_act_mx: x BF16 [M, K] (row stride ldx elements) -> q E4M3 codes
 * [M, K] (row stride K) and scale E8M0 bytes [M, K/32]. Per 1x32 block:
 * amax == 0 gives scale byte 0 and zero codes; otherwise the scale is
 * 2^(floor(log2 amax) - 8) clamped to [2^-127, 2^127] and each code is the
 * round-to-nearest-even E4M3 of x / scale, saturating at +-448.
 * Limits: K % 32 == 0, ldx >= K, ldx % 8 == 0.
 */
moe_status_t moe_quant_act_mx(const void* x_bf16, int M, int K, int ldx, uint8_t* q,
                              uint8_t* scale, moe_stream_t stream);

/* --------------------------------------------------------- weight prepack
 * The GEMMs stream each 128-row x 128-K weight tile as one contiguous 8 KB
 * block (one TMA request per tile instead of 128 strided 64-byte rows).
 * moe_prepack_weights_mx converts row-major packed E2M1 codes [E, N, K/2]
 * into [E][N/128][K/128][128 rows][64 bytes]: tile (nb, kb) of expert e holds
 * rows nb*128 .. nb*128+127, bytes kb*64 .. kb*64+63 of each row, rows in
 * order. Call once at weight-load time; the output is what fused_moe_* take
 * as w1 / w2. Limits: N % 128 == 0, K % 128 == 0; out must not alias w.
 */
size_t moe_prepacked_weight_bytes(int E, int N, int K);
moe_status_t moe_prepack_weights_mx(const uint8_t* w, int E, int N, int K, uint8_t* out,
                                    moe_stream_t stream);

/* moe_prepack_weights_a16w4: the weight prepack of the a16w4 calls (the
 * weights fused_moe_a16w4* take). The same tiles as moe_prepack_weights_mx,
 * and within every 32-bit word of eight E2M1 codes (code j in bits
 * 4j..4j+3, bit 3 the sign) the bits are moved so that the GEMM turns each
 * pair of codes into two BF16 values with a rotation and a mask: pair 0 =
 * w & P, pair 1 = rotr(w, 6) & P, pair 2 = rotr(w, 12) & P, pair 3 =
 * (rotr(w, 2) & PA) | (rotr(w, 10) & PB), with P = 0x81C081C0, PA =
 * 0x81808180, PB = 0x00400040; each BF16 half then holds its code's
 * mantissa, exponent and sign at bits 6, 7-8 and 15 (the E2M1 value times
 * 2^-126). Same size, limits and errors as moe_prepack_weights_mx. */
moe_status_t moe_prepack_weights_a16w4(const uint8_t* w, int E, int N, int K, uint8_t* out,
                                       moe_stream_t stream);

/* moe_dequant_a16w4 (diagnostic): the a16w4 GEMMs' dequantisation of whole
 * experts, run by the same device routine: w_packed from
 * moe_prepack_weights_a16w4, scale_packed from moe_prepack_scales_mx, out
 * BF16 [E, N, K] (device), element (e, n, k) = E2M1 code times 2^(s - 127)
 * of its block (OCP Microscaling Formats v1.0: MXFP4), exact wherever the
 * product is a BF16 number; products past the BF16 range are infinities,
 * and the NaN scale (255) gives infinities (NaN for the zero codes).
 * Limits and errors as moe_prepack_weights_mx. */
moe_status_t moe_dequant_a16w4(const uint8_t* w_packed, const uint8_t* scale_packed, int E, int N,
                               int K, void* out_bf16, moe_stream_t stream);

/* ---------------------------------------------------- weight scale prepack
 * The GEMMs read weight scales in 512-byte atoms. moe_prepack_scales_mx
 * converts row-major scales [E, N, K/32] into [E][N/128][K/128][512]: in the
 * atom of row block nb and K slab kb, the byte of row r (0..127) and 32-block
 * i (0..3) sits at (r % 32) * 16 + (r / 32) * 4 + i. Call once at weight-load
 * time; the output is what fused_moe_* take as w*_scale.
 * Limits: N % 128 == 0, K % 128 == 0.
 */
size_t moe_prepacked_scale_bytes(int E, int N, int K);
moe_status_t moe_prepack_scales_mx(const uint8_t* scale, int E, int N, int K, uint8_t* out,
                                   moe_stream_t stream);

/* ---------------------------------------------------------- fused layer
 * Workspace: fused_moe_workspace_bytes gives the size for the shape; the
 * caller allocates it (device, 256-byte aligned) and may reuse it for any
 * later call with the same or a smaller shape. Contents need no
 * initialisation. Two calls in flight on different streams need different
 * workspaces. Results are not bitwise reproducible from call to call: the
 * routing-weighted sum (and, for small calls, the parts of the tiles
 * that the split walk spreads over several CTAs) is added in FP32 by atomic
 * reductions whose order varies; the sorted lists are deterministic, and so
 * is the intermediate outside the split stage-1 tiles.
 */
typedef struct {
  int32_t block_m;       /* route block of both GEMMs (= sort block) */
  int32_t _pad;
  int64_t p_max;         /* sorted-list capacity */
  int64_t status_off;    /* int32[4]: [0] device status bits, [1] num_padded */
  int64_t expert_off_off;   /* int32 [E+1] */
  int64_t sorted_route_off; /* int32 [p_max] */
  int64_t sorted_w_off;     /* float [p_max] */
  int64_t block_expert_off; /* int32 [p_max/block_m] */
  int64_t route_pos_off;    /* int32 [M*topk] */
  int64_t sort_scratch_off; /* int32 per-CTA expert histograms of the sort */
  int64_t act_off;       /* a8w4: E4M3 [p_max, H] route rows; a16w4: BF16 [p_max, H];
                            rows of pad entries are not written */
  int64_t act_sf_off;    /* a8w4: scale atoms [p_max/block_m][H/128][ceil(block_m/128)][512] */
  int64_t inter_off;     /* a8w4: E4M3 [p_max, Ip]; a16w4: BF16 [p_max, Ip] */
  int64_t inter_sf_off;  /* a8w4: scale atoms [p_max/block_m][Ip/128][ceil(block_m/128)][512] */
  int64_t acc_off;       /* float [M, H] routing-weighted sum before BF16 rounding */
  int64_t split_part_off;   /* block_m <= 32: float [320][block_m][128] partial sums of
                               stage-1 tiles whose K range is split across CTAs; else empty */
  int64_t split_cnt_off;    /* int32 [320] arrival counters of those tiles; else empty */
  int64_t total_bytes;
} moe_ws_layout_t;

size_t fused_moe_workspace_bytes(int M, int H, int Ip, int E, int topk, int a16);
moe_status_t fused_moe_workspace_layout(int M, int H, int Ip, int E, int topk, int a16,
                                        moe_ws_layout_t* out /* host */);

/* fused_moe_a8w4: out = MoE(x) with FP8 activations and MXFP4 weights.
 *   x            BF16 [M, H]
 *   topk_ids     int32 [M, topk]  (ids outside [0, E) are dropped)
 *   topk_weights float [M, topk]
 *   w1           E2M1 codes of w1 [E, 2*Ip, H/2] (gate/up interleaved rows),
 *                prepacked by moe_prepack_weights_mx (N=2*Ip, K=H)
 *   w1_scale     scales of w1 prepacked by moe_prepack_scales_mx (N=2*Ip, K=H)
 *   w2           E2M1 codes of w2 [E, H, Ip/2] prepacked (N=H, K=Ip)
 *   w2_scale     scales of w2 prepacked (N=H, K=Ip)
 *   out          BF16 [M, H]
 * Ip is the stored (padded) intermediate size; padding rows/columns of the
 * weights must hold zero codes. Tokens without a local route get 0.
 * Limits: H % 128 == 0, Ip % 128 == 0, 1 <= E <= 512, 1 <= topk <= 16,
 * 0 <= M, M*topk <= 2^24.
 */
moe_status_t fused_moe_a8w4(const void* x, const int32_t* topk_ids, const float* topk_weights,
                            int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                            const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip, void* out,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/* fused_moe_a16w4: as fused_moe_a8w4 with BF16 activations (no activation
 * quantisation) and a BF16 intermediate; w1 / w2 come from
 * moe_prepack_weights_a16w4 (not moe_prepack_weights_mx). Otherwise the same
 * arguments and limits. */
moe_status_t fused_moe_a16w4(const void* x, const int32_t* topk_ids,
                             const float* topk_weights, int M, int H, int topk,
                             const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2,
                             const uint8_t* w2_scale, int E, int Ip, void* out, void* ws,
                             size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------- explicit route block (tuning)
 * The same calls with the route block chosen by the caller instead of the
 * library's rule (the sort block = the GEMMs' route tile, the knob a
 * per-token-bucket tuning table sets; AITER #5609 "Add DeepSeek V4.1 Flash
 * TP4 gfx950 MoE tuning", Commands run: the sort block must equal the GEMM
 * block). block_m: 0 for the library's rule, else one of 16, 32, 64, 128,
 * 256; any other value gives 0 bytes / MOE_ERR_UNSUPPORTED. A workspace and
 * its layout are valid only for the block_m they were sized with. The
 * result is the same for every block_m up to FP32 summation order. */
size_t fused_moe_workspace_bytes_bm(int M, int H, int Ip, int E, int topk, int a16, int block_m);
moe_status_t fused_moe_workspace_layout_bm(int M, int H, int Ip, int E, int topk, int a16,
                                           int block_m, moe_ws_layout_t* out /* host */);
moe_status_t fused_moe_a8w4_bm(const void* x, const int32_t* topk_ids, const float* topk_weights,
                               int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                               const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                               void* out, void* ws, size_t ws_bytes, int block_m,
                               moe_stream_t stream);
moe_status_t fused_moe_a16w4_bm(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                                const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                void* out, void* ws, size_t ws_bytes, int block_m,
                                moe_stream_t stream);

/* ------------------------------------------------ per-call configuration
 * The calls with every per-call tuning parameter the caller may set (the
 * rows of a per-token-bucket tuning table; AITER #5609 "Add DeepSeek V4.1
 * Flash TP4 gfx950 MoE tuning", Configuration: one configuration per
 * geometry and token bucket). A zero field is the library's choice.
 *   block_m    route block, as for the *_bm calls (0, 16, 32, 64, 128, 256);
 *              the workspace is sized by fused_moe_workspace_bytes_bm with it
 *   prefetch1  stage-1 weight L2 prefetch lead in 128-K weight tiles, 1..64
 *              (default a8w4 4, a16w4 8)
 *   prefetch2  the same for stage 2 (default a8w4 2, a16w4 8)
 *   split      at block_m <= 32: the GEMMs' split walk, in which every CTA
 *              takes an equal share of the tiles' K blocks (a tile spread
 *              over several CTAs is computed in parts) when there are fewer
 *              than 8 waves of tiles, and whole tiles otherwise. 0 = the
 *              library's choice (the split walk), 1 = the split walk,
 *              2 = whole tiles only.
 * Out-of-range values give MOE_ERR_UNSUPPORTED. cfg NULL = all defaults.
 * The result does not depend on the prefetch leads (they only move weight
 * tiles into L2 earlier or later); the split walk changes the order of FP32
 * additions only. */
typedef struct {
  int32_t block_m;
  int32_t prefetch1;
  int32_t prefetch2;
  int32_t split;
} moe_call_config_t;
moe_status_t fused_moe_a8w4_cfg(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                                const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                void* out, void* ws, size_t ws_bytes,
                                const moe_call_config_t* cfg /* host */, moe_stream_t stream);
moe_status_t fused_moe_a16w4_cfg(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                 int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                                 const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                 void* out, void* ws, size_t ws_bytes,
                                 const moe_call_config_t* cfg /* host */, moe_stream_t stream);

/* ------------------------------------------------------- gated calls
 * fused_moe_a8w4_gated / fused_moe_a16w4_gated: the fused calls with the
 * gating in front (the pages time the local MoE "including gating", AITER
 * #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the
 * measured runtime). The routing is that of moe_router_topk on
 * router_logits (float32 [M, E_route], row stride ld >= E_route): per token
 * the topk largest logits (ties to the lower expert), weights = softmax over
 * the picks, and with shared_id >= 0 n_shared last columns shared_id, ...,
 * shared_id + n_shared - 1 of weight 1.0. It is written to topk_ids (int32)
 * / topk_weights (float) [M, k'] with k' = topk + n_shared (0 shared columns
 * when shared_id < 0), caller-allocated device buffers, and the
 * layer then computes exactly what fused_moe_* computes with those ids and
 * weights and topk = k' (ids outside [0, E) are dropped; expert-parallel
 * shards pass the global logits). Up to 256 routes (M * k') the gating runs
 * inside the call's first kernel, together with the sort and the gather;
 * beyond that the gating kernel is its own launch.
 * Workspace: fused_moe_workspace_bytes(M, H, Ip, E, k', a16).
 * Errors: MOE_ERR_INVALID_ARG for ld < E_route, topk outside [1, E_route],
 * shared_id >= 0 with shared_id < E_route, n_shared < 1 or shared_id +
 * n_shared > 512, NULL logits / id / weight buffers
 * with M > 0, and the errors of fused_moe_a8w4; MOE_ERR_UNSUPPORTED for
 * E_route > 512 or k' > 16; MOE_ERR_ALIGNMENT for pointers not 256-byte
 * aligned. All before any launch.
 */
moe_status_t fused_moe_a8w4_gated(const void* x, const float* router_logits, int ld, int E_route,
                                  int topk, int shared_id, int n_shared, int M, int H,
                                  const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2,
                                  const uint8_t* w2_scale, int E, int Ip, void* out,
                                  int32_t* topk_ids, float* topk_weights, void* ws,
                                  size_t ws_bytes, moe_stream_t stream);
moe_status_t fused_moe_a16w4_gated(const void* x, const float* router_logits, int ld,
                                   int E_route, int topk, int shared_id, int n_shared, int M,
                                   int H, const uint8_t* w1, const uint8_t* w1_scale,
                                   const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                   void* out, int32_t* topk_ids, float* topk_weights, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------ no-allocation variant
 * fused_moe_a8w4_noalloc: fused_moe_a8w4 without a caller workspace. The
 * pages have no counterpart of this entry point; it exists for callers that
 * cannot hand the library scratch memory, such as a plugin inside an engine
 * that owns every device allocation and gives its plugins no way to ask for
 * more, or a latency-critical path that may not call a device allocator.
 * The caller still provides every input, the weights and the output.
 *
 * The scratch is one static device array of MOE_NOALLOC_WORKSPACE_BYTES
 * inside this library; each GPU that loads the library keeps it until the
 * process exits. Shapes whose fused_moe_workspace_bytes() exceeds that size
 * are rejected with MOE_ERR_WORKSPACE before anything is launched (with the
 * current workspace layout that is up to 19 tokens at H=5120, Ip=640, 384
 * experts, top-6, and up to 38 tokens at 128 experts, top-3).
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any
 * stream capture on the device. The cached address is that of the device
 * context current at the first call: after cudaDeviceReset on a device this
 * entry point (and moe_noalloc_status) must not be used on that device
 * again in the same process. All calls share the one array and it keeps
 * the previous call's contents (no part of it needs to start at zero), so
 * calls that can overlap on the GPU (different streams, or different host
 * threads) race on it: serialise them. Arguments, limits, layouts and errors
 * are otherwise those of fused_moe_a8w4; the device status words that
 * fused_moe_a8w4 leaves in the caller's workspace are read with
 * moe_noalloc_status.
 */
#define MOE_NOALLOC_WORKSPACE_BYTES (16u << 20)
moe_status_t fused_moe_a8w4_noalloc(const void* x, const int32_t* topk_ids,
                                    const float* topk_weights, int M, int H, int topk,
                                    const uint8_t* w1, const uint8_t* w1_scale,
                                    const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                    void* out, moe_stream_t stream);

/* moe_noalloc_status: the device-side status of the last
 * fused_moe_a8w4_noalloc call on the current device. Enqueues, on `stream`,
 * a device-to-device copy of the scratch array's status words (int32[4]:
 * [0] device status bits, decoded by moe_decode_device_status; [1] the
 * padded route count P) into status_out, a caller-owned device buffer of 16
 * bytes, 16-byte aligned. Allocates nothing. Read it after the call it
 * reports on has completed on that stream (same stream order, or a sync).
 * MOE_ERR_INVALID_ARG for a NULL pointer, MOE_ERR_ALIGNMENT for a
 * misaligned one, MOE_ERR_CUDA if the copy cannot be enqueued. */
moe_status_t moe_noalloc_status(int32_t* status_out, moe_stream_t stream);

/* --------------------------------------------------------- kernel timing
 * For benchmarks and profiling. While enabled, every fused_moe_* call records
 * a CUDA event right before and right after each of its kernel launches, on
 * the call's stream (slot 0 sort, 1 activation gather/quant, 2 stage-1 GEMM,
 * 3 stage-2 GEMM, 4 BF16 finalise). moe_profile_collect waits for those
 * events, adds each slot's elapsed milliseconds into kernel_ms[slot] (an
 * array of MOE_PROFILE_SLOTS doubles, host), writes the number of calls
 * measured to *n_calls and forgets them. Off by default; the events are
 * created on first use and kept. Up to 1024 calls may be pending; later
 * calls are not recorded. Not thread-safe; do not enable it while capturing
 * a CUDA graph.
 */
#define MOE_PROFILE_SLOTS 5
moe_status_t moe_profile_enable(int enable);
moe_status_t moe_profile_collect(double* kernel_ms, int32_t* n_calls);

/* Decode the status word copied from the workspace (host value) into a
 * moe_status_t: MOE_OK; MOE_ERR_TIMEOUT if a device wait gave up (bit 0);
 * MOE_ERR_DEVICE_CHECK if a GEMM met a route block whose expert id was
 * outside [0, E) (bit 1; it then used expert 0 for that block, so no access
 * left the weight arrays, and the output is not valid). */
moe_status_t moe_decode_device_status(int32_t status_word);

/* Self-test of the device-side failure reporting: one kernel waits, with the
 * same bounded wait every kernel of the layer uses, on a barrier that
 * nothing completes; after timeout_us (1 .. 1e6) of global time the wait
 * gives up, ORs the timeout bit into status[0] and the kernel writes
 * status[1] = 1 and returns (2 would mean the wait completed). status: device
 * int32[2], zeroed by the caller, 256-byte aligned. The GPU is neither hung
 * nor faulted and the context stays usable. MOE_ERR_INVALID_ARG /
 * MOE_ERR_ALIGNMENT before any launch. */
moe_status_t moe_debug_wait_selftest(int32_t* status, int timeout_us, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MX_H */
