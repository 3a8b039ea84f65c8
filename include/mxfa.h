/*
 * mxfa.h -- C ABI of libmxfa: MXFP8 block-scaled FlashAttention (forward and
 * backward) for NVIDIA GB300 (sm_103a), with its quantizers and the fused
 * RMSNorm+Quantize producer.
 *
 * Sources for what each call computes (web pages on one subject):
 *  [MX]   "Low-Precision FlashAttention-4: End-to-End Block-Scaled Attention
 *         on Blackwell" (kongchang.com), section "Why MXFP8" -- OCP MX: 32
 *         elements share one power-of-two (E8M0) scale, E4M3 payload.
 *  [TMEM] "MXFP8 FlashAttention-4 Hits 2.85 Petaflops in Meta's Production
 *         Training" (andresseo.expert), section "Inside the TMEM Bargain and
 *         Zero-Gather Jagged Pipeline" -- online P / dS quantization, square
 *         32x32 blocks for Q, K, dO in the backward pass, dQ reduction in
 *         FP16 with static scaling, split addressing for jagged inputs,
 *         fused RMSNorm / GEMM producers.
 *  [KDIM] "Meta's MXFP8 FlashAttention-4 kernel, tackling TMEM scale-factor
 *         constraints, hits up to 1.6x over BF16" (theclarity.today),
 *         paragraphs 1-3 -- scales along the MMA K dimension (D for Q and K,
 *         N for V); scales padded and permuted to 128-aligned layouts for TMA.
 *  [ITEMS] "Meta's FlashAttention-4 Achieves 2.85 PF/s with MXFP8 on Blackwell
 *         GPUs" (brifing.si), items 5 (jagged), 6 (backward), 7 (fused
 *         producers).
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises (except mxfa_get_device_status).
 *    Work is enqueued on the caller's stream (a cudaStream_t; 0 = legacy).
 *  - Attention tensors are token-major: x[token][head][d] with d contiguous
 *    (dense [B][S][H][D] is the varlen layout with B sequences of length S).
 *    D must be 128.
 *  - Payload pointers, scale pointers and bf16 outputs must be 16-byte
 *    aligned (else MXFA_ERR_MISALIGNED).
 *  - Arguments are checked before any launch; launch failures are reported
 *    as MXFA_ERR_CUDA.  Device-side failures (a bounded wait that expired,
 *    an index check that skipped an access) are recorded in a status word
 *    read by mxfa_get_device_status.  Nothing aborts the process.
 *
 * Scale-factor layouts
 *  compact (one E8M0 byte per block, logical order):
 *    ROW  [tokens][H*D/32]            1x32 along d
 *    COL  [sum ceil(len/32)][H*D]     32x1 along the tokens of a sequence
 *    SQ   [sum ceil(len/32)][H*D/32]  32x32 within a head
 *  packed (what the attention kernels read; rows padded per sequence to a
 *  multiple of 128 with value 0x7F, i.e. 2^0):
 *    tiles = sum over sequences of ceil(len/128); tile t of head h is entry
 *    (t * H + h).
 *    ROW  512-byte atom per entry: byte (r%32)*16 + (r/32)*4 + k for token r
 *         of the tile and d-block k  (the tensor core's 128x4 scale layout)
 *    COL  512-byte atom per entry: byte (d%32)*16 + (d/32)*4 + k for column d
 *         and 32-token block k of the tile
 *    SQ   16 bytes per entry: byte 4*k + c for token block k and d-block c
 */
#ifndef MXFA_H
#define MXFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mxfa_stream_t; /* same type as cudaStream_t */

typedef enum {
  MXFA_OK = 0,
  MXFA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum        */
  MXFA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. D!=128) */
  MXFA_ERR_MISALIGNED = 3,    /* pointer not 16-byte aligned             */
  MXFA_ERR_WORKSPACE_TOO_SMALL = 4,
  MXFA_ERR_CUDA = 5,          /* a CUDA call or kernel launch failed     */
  MXFA_ERR_TIMEOUT = 6,       /* a kernel's bounded wait expired         */
  MXFA_ERR_DEVICE_INDEX = 7   /* a kernel's index check skipped an access */
} mxfa_status;

typedef enum {
  MXFA_BLK_ROW = 0, /* 1x32 along d (MMA K = D: Q, K forward; V backward)    */
  MXFA_BLK_COL = 1, /* 32x1 along tokens of a sequence (MMA K = N: V forward) */
  MXFA_BLK_SQ = 2   /* 32x32, transpose-invariant (Q, K, dO backward)         */
} mxfa_block;

/* An MXFP8 operand as the attention kernels read it: E4M3 payload in the
 * source layout (compact, never padded) and E8M0 scales in the packed
 * layout of its block kind. */
typedef struct {
  const uint8_t* data;
  const uint8_t* sf;
} mxfa_mx;

/* Outputs of a quantizing call; sf_compact and sf_packed may be NULL. */
typedef struct {
  uint8_t* data;
  uint8_t* sf_compact;
  uint8_t* sf_packed;
} mxfa_mx_out;

/* The forward kernel moves its running row maximum only when it grows by
 * more than this many log2 units (O and l keep the stale maximum exactly). */
#define MXFA_FWD_RESCALE_THRESHOLD 8.0f

/* Options of the *_opts attention calls (the plain calls use the defaults).
 *  rescale_threshold  forward only: the running row maximum moves when it
 *          grows by more than this (log2 units, 0 <= t <= 8); 0 rescales at
 *          every increase.  P~ = 2^(s' - m) then stays below 2^t.  Default
 *          MXFA_FWD_RESCALE_THRESHOLD.
 *  p_scale MXFA_P_SCALE_BLOCK (default): each 32-element block of P gets the
 *          E8M0 scale of its own maximum (OCP rule).  MXFA_P_SCALE_CONST: one
 *          constant scale for every block ([ITEMS] item 4: constant scaling
 *          of softmax outputs, which lie in a known range): forward
 *          2^(ceil(t) - 8), so the largest possible P~, 2^ceil(t), maps to
 *          256 <= 448; backward 2^-8 (P <= 1 maps to <= 256).  Values below
 *          2^-9 of the scale round to zero. */
#define MXFA_P_SCALE_BLOCK 0
#define MXFA_P_SCALE_CONST 1
typedef struct {
  float rescale_threshold;
  int p_scale;
} mxfa_attn_opts;

const char* mxfa_status_string(mxfa_status s);
int mxfa_version(void);

/* Number of packed tiles: sum over sequences of ceil(len/128).  cu_seqlens
 * here is a HOST array of nseq+1 offsets; NULL means nseq sequences of
 * seqlen tokens.  Returns -1 on bad input. */
int64_t mxfa_packed_tiles(const int32_t* cu_seqlens_host, int nseq, int seqlen);
/* Bytes of a packed scale tensor for `tiles` packed tiles and H heads. */
size_t mxfa_sf_packed_bytes(mxfa_block blk, int64_t tiles, int H);

/* mxfa_quantize -- bf16 -> E4M3 payload + E8M0 scales ([MX]; orientation
 * per [KDIM] and [TMEM]).
 *  x          bf16 [tokens][H][D], D = 128
 *  blk        block kind
 *  cu_seqlens DEVICE int32[nseq+1] sequence offsets, or NULL for nseq
 *             sequences of max_seqlen tokens each (tokens = nseq*max_seqlen)
 *  max_seqlen longest sequence (sizes the grid)
 *  packed_tiles  mxfa_packed_tiles() of the same sequences (bounds the
 *             packed output; ignored when out->sf_packed is NULL)
 *  out        payload [tokens][H][D] and the compact and/or packed scales
 * Scale: floor(log2 amax) - 8 clamped to [0, 254]; payload RNE, saturating
 * at 448; a block holding Inf/NaN gets scale 0xFF and payload 0x7F. */
mxfa_status mxfa_quantize(const void* x, int64_t tokens, int H, int D, mxfa_block blk,
                          const int32_t* cu_seqlens, int nseq, int max_seqlen,
                          int64_t packed_tiles, const mxfa_mx_out* out, mxfa_stream_t stream);

/* mxfa_quantize_dual -- one read of x, two layouts: blk (MXFA_BLK_COL or
 * MXFA_BLK_SQ) into out, and MXFA_BLK_ROW into out_row, each byte for byte as
 * mxfa_quantize would write it ([ITEMS] item 7: quantization fused so that no
 * separate pass reads the tensor again).  COL + ROW serves V (forward, then
 * backward); SQ + ROW serves Q and K (backward, then forward).  Arguments as
 * mxfa_quantize; out_row and its payload are required, its scale pointers
 * nullable; another blk is MXFA_ERR_INVALID_ARG. */
mxfa_status mxfa_quantize_dual(const void* x, int64_t tokens, int H, int D, mxfa_block blk,
                               const int32_t* cu_seqlens, int nseq, int max_seqlen,
                               int64_t packed_tiles, const mxfa_mx_out* out,
                               const mxfa_mx_out* out_row, mxfa_stream_t stream);

/* mxfa_sf_pack -- compact scales -> packed scales for the same block kind,
 * values unchanged, padding rows 0x7F ([KDIM] paragraph 3, [ITEMS] item 5:
 * only the scale factors are scattered and padded; payload stays compact).
 * Arguments as mxfa_quantize. */
mxfa_status mxfa_sf_pack(const uint8_t* sf_compact, int64_t tokens, int H, int D, mxfa_block blk,
                         const int32_t* cu_seqlens, int nseq, int max_seqlen,
                         int64_t packed_tiles, uint8_t* sf_packed, mxfa_stream_t stream);

/* mxfa_sf_unpack -- packed scales -> compact scales: the inverse of
 * mxfa_sf_pack for every real row / block (padding bytes are not read).
 * It gives tests and tools a C-ABI round trip of the packed layout that the
 * tensor core reads; it is not on the training path.  Arguments as
 * mxfa_sf_pack with the roles of the two scale buffers exchanged. */
mxfa_status mxfa_sf_unpack(const uint8_t* sf_packed, int64_t tokens, int H, int D, mxfa_block blk,
                           const int32_t* cu_seqlens, int nseq, int max_seqlen,
                           int64_t packed_tiles, uint8_t* sf_compact, mxfa_stream_t stream);

/* mxfa_fwd -- dense forward ([KDIM] paragraphs 1-2, [TMEM]).
 *  q, k       ROW-quantized payload [B][S][H][128] + packed ROW scales
 *  v          COL-quantized payload + packed COL scales
 *  causal     mask key > query
 *  o          bf16 [B][S][H][128] (output)
 *  lse        fp32 [B][H][S] natural-log log-sum-exp (output)
 * P is quantized per 32 keys in registers; the row sum is taken before. */
mxfa_status mxfa_fwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, int B, int S, int H,
                     int D, float softmax_scale, int causal, void* o, float* lse,
                     mxfa_stream_t stream);

/* mxfa_varlen_fwd -- jagged forward ([TMEM] split addressing, [ITEMS] 5).
 *  cu_seqlens_q/k  DEVICE int32[nseq+1]; q/o/lse follow cu_seqlens_q,
 *                  k/v follow cu_seqlens_k.  Lengths may be 0: a query
 *                  sequence whose key sequence is empty gets O = 0 and
 *                  lse = -inf (the empty softmax sum); an empty query
 *                  sequence writes nothing.  max_seqlen_k must be >= 1.
 *  ptiles_q/k      mxfa_packed_tiles() of the query / key sequences
 *  lse             fp32 [H][total_q]
 *  causal          top-left aligned (key index > query index masked) */
mxfa_status mxfa_varlen_fwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, int64_t total_q, int64_t total_k,
                            int64_t ptiles_q, int64_t ptiles_k, int H, int D, float softmax_scale,
                            int causal, void* o, float* lse, mxfa_stream_t stream);

/* mxfa_fwd_mxo, mxfa_varlen_fwd_mxo -- the forward passes above that also
 * emit O as MXFP8 for the output projection ([KDIM] paragraph 4: fused
 * producer and output epilogues).  The bf16 O they write is quantized in
 * 1x32 blocks along D, byte for byte as mxfa_quantize(MXFA_BLK_ROW)
 * quantizes that bf16 O:
 *  o_mx->data        E4M3 [tokens][H][128] (required, 16-byte aligned)
 *  o_mx->sf_compact  E8M0 [tokens][H * 4] (nullable, 4-byte aligned)
 *  o_mx->sf_packed   packed ROW atoms, ptiles_q * H * 512 bytes, rows past
 *                    a sequence's end 0x7F (nullable, 16-byte aligned)
 * Other arguments and errors as mxfa_fwd / mxfa_varlen_fwd; o_mx NULL is
 * MXFA_ERR_INVALID_ARG. */
mxfa_status mxfa_fwd_mxo(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, int B, int S, int H,
                         int D, float softmax_scale, int causal, void* o, float* lse,
                         const mxfa_mx_out* o_mx, mxfa_stream_t stream);
mxfa_status mxfa_varlen_fwd_mxo(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                                int max_seqlen_q, int max_seqlen_k, int64_t total_q,
                                int64_t total_k, int64_t ptiles_q, int64_t ptiles_k, int H, int D,
                                float softmax_scale, int causal, void* o, float* lse,
                                const mxfa_mx_out* o_mx, mxfa_stream_t stream);

/* mxfa_fwd_opts, mxfa_varlen_fwd_opts -- mxfa_fwd / mxfa_varlen_fwd with
 * options (see mxfa_attn_opts; NULL = defaults).  A threshold outside
 * [0, 8] or an unknown p_scale is MXFA_ERR_INVALID_ARG. */
mxfa_status mxfa_fwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, int B, int S, int H,
                          int D, float softmax_scale, int causal, const mxfa_attn_opts* opts,
                          void* o, float* lse, mxfa_stream_t stream);
mxfa_status mxfa_varlen_fwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                                 int max_seqlen_q, int max_seqlen_k, int64_t total_q,
                                 int64_t total_k, int64_t ptiles_q, int64_t ptiles_k, int H, int D,
                                 float softmax_scale, int causal, const mxfa_attn_opts* opts,
                                 void* o, float* lse, mxfa_stream_t stream);

/* Workspace of the backward pass for total_q query tokens in nseq sequences:
 * one 2560-byte record per (64-query tile, head) -- the tile's scale atoms,
 * lse * log2(e) and Delta = rowsum(dO^ * O) -- for at most
 * ceil(total_q / 64) + nseq tiles, followed by the dQ accumulator
 * ([total_q][H][128], fp32 when dq_mode = 0, fp16 when 1). */
size_t mxfa_bwd_workspace_size(int64_t total_q, int nseq, int H, int D, int dq_mode);

/* mxfa_bwd -- dense backward, five GEMMs with recompute ([TMEM], [ITEMS] 6).
 *  q, k, dO   SQ-quantized payload + packed SQ scales (32x32 blocks serve
 *             both GEMM orientations)
 *  v          ROW-quantized payload + packed ROW scales
 *  o, dout    bf16 O and dO [B][S][H][128];  lse fp32 [B][H][S] from mxfa_fwd.
 *             Delta = rowsum(dO^ * O) takes the dequantized square-block dO^
 *             of dout_mx (the operand that also enters dP), so dout itself
 *             is checked but not read
 *  dq_mode    0: dQ reduced in fp32;  1: fp16 with static scale
 *             dq_static_scale (a power of two; partials are multiplied by it
 *             before the fp16 reduction and divided after)
 *  dq, dk, dv bf16 outputs [B][S][H][128]
 *  ws         caller-owned workspace of mxfa_bwd_workspace_size() bytes
 * P is recomputed from the square-block Q, K and lse, quantized 1x32 along
 * queries for dV; dS = P (dP - Delta) is quantized in 32x32 blocks. */
mxfa_status mxfa_bwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dout_mx,
                     const void* o, const void* dout, const float* lse, int B, int S, int H, int D,
                     float softmax_scale, int causal, int dq_mode, float dq_static_scale, void* dq,
                     void* dk, void* dv, void* ws, size_t ws_bytes, mxfa_stream_t stream);

/* mxfa_varlen_bwd -- jagged backward; arguments as mxfa_varlen_fwd and
 * mxfa_bwd (lse [H][total_q]).  Keys of a sequence with no queries get
 * dK = dV = 0; queries of a sequence with no keys get dQ = 0. */
mxfa_status mxfa_varlen_bwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                            const mxfa_mx* dout_mx, const void* o, const void* dout, const float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, int64_t total_q, int64_t total_k,
                            int64_t ptiles_q, int64_t ptiles_k, int H, int D, float softmax_scale,
                            int causal, int dq_mode, float dq_static_scale, void* dq, void* dk,
                            void* dv, void* ws, size_t ws_bytes, mxfa_stream_t stream);

/* mxfa_bwd_opts, mxfa_varlen_bwd_opts -- mxfa_bwd / mxfa_varlen_bwd with
 * options (see mxfa_attn_opts; NULL = defaults; the backward reads only
 * p_scale, which selects the block or constant scale of its P^T). */
mxfa_status mxfa_bwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                          const mxfa_mx* dout_mx, const void* o, const void* dout, const float* lse,
                          int B, int S, int H, int D, float softmax_scale, int causal,
                          const mxfa_attn_opts* opts, int dq_mode, float dq_static_scale, void* dq,
                          void* dk, void* dv, void* ws, size_t ws_bytes, mxfa_stream_t stream);
mxfa_status mxfa_varlen_bwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                 const mxfa_mx* dout_mx, const void* o, const void* dout,
                                 const float* lse, const int32_t* cu_seqlens_q,
                                 const int32_t* cu_seqlens_k, int nseq, int max_seqlen_q,
                                 int max_seqlen_k, int64_t total_q, int64_t total_k,
                                 int64_t ptiles_q, int64_t ptiles_k, int H, int D,
                                 float softmax_scale, int causal, const mxfa_attn_opts* opts,
                                 int dq_mode, float dq_static_scale, void* dq, void* dk, void* dv,
                                 void* ws, size_t ws_bytes, mxfa_stream_t stream);

/* mxfa_bwd_mxg, mxfa_varlen_bwd_mxg -- the backward passes above that also
 * emit the gradients as MXFP8 ([TMEM] page, section "What the Benchmarks
 * Show About Low-Precision Training": quantized gradients instead of bf16).
 * Each bf16 gradient they write is quantized in 1x32 blocks along D, byte
 * for byte as mxfa_quantize(MXFA_BLK_ROW) quantizes it.  dq_mx, dk_mx, dv_mx
 * are each nullable; for each given one:
 *  data        E4M3 [tokens][H][128] (required, 16-byte aligned)
 *  sf_compact  E8M0 [tokens][H * 4] (nullable, 4-byte aligned; required for
 *              dq_mx when its sf_packed is given)
 *  sf_packed   packed ROW atoms, ptiles * H * 512 bytes, rows past a
 *              sequence's end 0x7F (nullable, 16-byte aligned)
 * dK and dV are quantized in the kernel's epilogue, dQ in its final pass
 * (plus one scale-packing pass when dq_mx->sf_packed is given).  Other
 * arguments and errors as mxfa_bwd / mxfa_varlen_bwd. */
mxfa_status mxfa_bwd_mxg(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                         const mxfa_mx* dout_mx, const void* o, const void* dout, const float* lse,
                         int B, int S, int H, int D, float softmax_scale, int causal, int dq_mode,
                         float dq_static_scale, void* dq, void* dk, void* dv, void* ws,
                         size_t ws_bytes, const mxfa_mx_out* dq_mx, const mxfa_mx_out* dk_mx,
                         const mxfa_mx_out* dv_mx, mxfa_stream_t stream);
mxfa_status mxfa_varlen_bwd_mxg(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                const mxfa_mx* dout_mx, const void* o, const void* dout,
                                const float* lse, const int32_t* cu_seqlens_q,
                                const int32_t* cu_seqlens_k, int nseq, int max_seqlen_q,
                                int max_seqlen_k, int64_t total_q, int64_t total_k,
                                int64_t ptiles_q, int64_t ptiles_k, int H, int D,
                                float softmax_scale, int causal, int dq_mode, float dq_static_scale,
                                void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                                const mxfa_mx_out* dq_mx, const mxfa_mx_out* dk_mx,
                                const mxfa_mx_out* dv_mx, mxfa_stream_t stream);

/* mxfa_rmsnorm_quant -- fused RMSNorm + MX quantization in one pass
 * ([TMEM] "fused producers", [ITEMS] item 7: FP8 out with dual scale layouts).
 *  x      bf16 [T][C], C in {256, 512, 1024, 2048}
 *  gamma  fp32 [C]
 *  y = (x * r) * gamma, r = 1/sqrt(mean(x^2) + eps), fp32, each operation
 *  correctly rounded; the sum of squares runs in a fixed order: lane l of a
 *  warp owns columns 8l + 256k + j, adds their squares k-outer, j-inner, then
 *  a butterfly over lane distances 16, 8, 4, 2, 1.
 *  seg_len  column and square blocks are anchored every seg_len rows
 *           (a multiple of 32; a multiple of 128 dividing T when packed
 *           scales are requested)
 *  H        head split of C for the packed layouts (C = H * 128)
 *  row/col/sq  outputs for 1x32, 32x1 and 32x32 blocks; each may be NULL
 *           (at least one must be given). */
mxfa_status mxfa_rmsnorm_quant(const void* x, const float* gamma, int64_t T, int64_t C, float eps,
                               int seg_len, int H, const mxfa_mx_out* row, const mxfa_mx_out* col,
                               const mxfa_mx_out* sq, mxfa_stream_t stream);

/* mxfa_bwd_noalloc -- mxfa_bwd for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call: it is an interface
 * addition of this library.
 *  For code that must not call cudaMalloc (allocator or memory-pool hooks,
 *  runtimes that forbid device allocation after start-up, bindings without a
 *  device allocator), the workspace comes from a scratch array compiled into
 *  the library (mxfa_bwd_noalloc_scratch_bytes() = 32 MiB, 256-byte aligned,
 *  held by every GPU that loads the library until the process exits).  The
 *  call allocates nothing; inputs and outputs are as for mxfa_bwd.
 *  The first call on each device looks up the array's device address
 *  (cudaGetSymbolAddress, with that device current) and caches it: make that
 *  first call before any stream capture.
 *  Problems whose workspace (mxfa_bwd_workspace_size) exceeds the array are
 *  rejected with MXFA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *  All calls share the one array and it keeps the last call's contents (the
 *  backward pass clears what must start at zero); calls that overlap on the
 *  GPU, e.g. on two streams, race on it. */
mxfa_status mxfa_bwd_noalloc(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                             const mxfa_mx* dout_mx, const void* o, const void* dout,
                             const float* lse, int B, int S, int H, int D, float softmax_scale,
                             int causal, int dq_mode, float dq_static_scale, void* dq, void* dk,
                             void* dv, mxfa_stream_t stream);
size_t mxfa_bwd_noalloc_scratch_bytes(void);

/* mxfa_gemm_quant -- projection GEMM with the quantization fused into its
 * epilogue ([TMEM] "fused producers": projection GEMM epilogues emit FP8;
 * [ITEMS] item 7: GEMM+Quantize with dual scale-factor layouts in one pass).
 *  a   ROW-quantized A [M][K] (payload, and packed ROW scales with K / 128
 *      column groups, i.e. mxfa_quantize(MXFA_BLK_ROW) of a bf16 [M][K/128][128])
 *  b   ROW-quantized B [N][K] likewise (a weight stored [out][in])
 *  Y = A B^T (dequantized operands, fp32 accumulation), written as
 *  y_bf16  bf16 [M][N] (nullable)
 *  y_row   MXFP8 of Y in 1x32 blocks along N: payload [M][N], compact scales
 *          [M][N / 32], packed ROW atoms of (128-row tile, 128-column group),
 *          as mxfa_quantize(MXFA_BLK_ROW) lays them out for Y seen as
 *          [M][N / 128][128] (nullable; its scale pointers nullable)
 *  y_col   MXFP8 of Y in 32x1 blocks along M (blocks start at multiples of
 *          32 rows): payload [M][N], compact scales [M / 32][N], packed COL
 *          atoms (nullable; its scale pointers nullable)
 *  At least one output must be given.  M, N, K multiples of 128
 *  (else MXFA_ERR_UNSUPPORTED).  Each output block is quantized with the OCP
 *  rule of mxfa_quantize from the fp32 value of Y (not from its bf16 copy). */
mxfa_status mxfa_gemm_quant(const mxfa_mx* a, const mxfa_mx* b, int64_t M, int64_t N, int64_t K,
                            void* y_bf16, const mxfa_mx_out* y_row, const mxfa_mx_out* y_col,
                            mxfa_stream_t stream);

/* Lower-precision formats -- the next formats the pages name ([ITEMS] item
 * 12: MXFP6 and MXFP4; [KDIM] paragraph 1: Blackwell's block-scaled MMA runs
 * MXFP8, MXFP6, MXFP4 and NVFP4).
 * mxfa_quantize_lowp -- bf16 x[rows][cols] -> codes in 1x32 blocks along the
 * columns with E8M0 scales
 * (MXFP4 = E2M1, max 6, emax 2; MXFP6 = E2M3, max 7.5, emax 2, or E3M2, max
 * 28, emax 4: scale = floor(log2 amax) - emax, clamped to [0, 254]; codes
 * nearest-even, saturating; a block holding Inf / NaN gets scale 0xFF and
 * codes 0), or NVFP4 in 1x16 blocks: fp32 tensor scale st = amax / 2688
 * (448 * 6; 1 for an all-zero tensor), written to *tensor_scale (DEVICE),
 * E4M3 block scales E4M3(amax_block / (6 st)) and E2M1 codes of
 * x / (scale * st), every step one correctly rounded fp32 operation (NVFP4
 * inputs must be finite).
 *  q          [rows][cols] bytes: with MXFA_LOWP_CODES one code per byte in
 *             the low bits; with MXFA_LOWP_MMA (MX formats) the form the
 *             block-scaled MMA reads sub-byte operands in from shared memory:
 *             each run of 16 codes packed little-endian (code j at bit 4j for
 *             FP4, 6j for FP6) in the first 8 / 12 bytes of a 16-byte group,
 *             the rest zero -- still one byte of storage per element
 *  sf         scales [rows][cols / 32] (MX) or [rows][cols / 16] (NVFP4)
 *  sf_packed  MX only, nullable: packed atoms per (128-row tile, 128-column
 *             group) as the GEMM reads them (rows, cols multiples of 128)
 * cols must be a multiple of 32 (MX) or 16 (NVFP4). */
#define MXFA_LOWP_MXFP4 0
#define MXFA_LOWP_MXFP6_E2M3 1
#define MXFA_LOWP_MXFP6_E3M2 2
#define MXFA_LOWP_NVFP4 3
#define MXFA_LOWP_CODES 0
#define MXFA_LOWP_MMA 1
mxfa_status mxfa_quantize_lowp(const void* x, int64_t rows, int cols, int fmt, int q_layout, uint8_t* q,
                               uint8_t* sf, uint8_t* sf_packed, float* tensor_scale, mxfa_stream_t stream);

/* mxfa_gemm_quant_fmt -- mxfa_gemm_quant with the element format of each
 * operand: MXFA_ELEM_E4M3 (MXFP8), or MXFP6 / MXFP4 operands from
 * mxfa_quantize_lowp (MXFA_LOWP_MMA layout, packed scale atoms), which the tensor
 * core's mixed-format block-scaled MMA reads at the MXFP8 rate.  The output
 * options are those of mxfa_gemm_quant. */
#define MXFA_ELEM_E4M3 0
#define MXFA_ELEM_E2M3 1
#define MXFA_ELEM_E3M2 2
#define MXFA_ELEM_E2M1 3
mxfa_status mxfa_gemm_quant_fmt(const mxfa_mx* a, int a_fmt, const mxfa_mx* b, int b_fmt, int64_t M,
                                int64_t N, int64_t K, void* y_bf16, const mxfa_mx_out* y_row,
                                const mxfa_mx_out* y_col, mxfa_stream_t stream);

/* mxfa_tensor_peak_probe -- `ctas` CTAs (one per SM at most) each issue
 * `iters` x 4 back-to-back block-scaled MMAs (M = 128, N = 256, K = 32, E4M3,
 * operands resident in shared memory) and write the SM clock cycles they took
 * to cycles[ctas] (DEVICE, 8-byte aligned).  The pages have no counterpart: it
 * measures this GPU's dense MXFP8 tensor-pipe peak, the denominator of the
 * benchmark's roofline fractions (MACs per CTA = iters * 4 * 128 * 256 * 32). */
mxfa_status mxfa_tensor_peak_probe(int iters, int ctas, unsigned long long* cycles, mxfa_stream_t stream);

/* Synchronise `stream`, then return and clear the device status words:
 * MXFA_OK, MXFA_ERR_TIMEOUT or MXFA_ERR_DEVICE_INDEX (bit flags also in
 * *flags when flags is not NULL: 1 timeout, 2 index). */
mxfa_status mxfa_get_device_status(mxfa_stream_t stream, unsigned* flags);

#ifdef __cplusplus
}
#endif
#endif /* MXFA_H */
