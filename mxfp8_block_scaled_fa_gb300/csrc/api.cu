// api.cu -- the C ABI (include/mxfa.h): argument checks, TMA descriptors and
// kernel launches.  No allocation, no synchronisation on the hot path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mxfa.h"
#include "mxfa_internal.h"

using namespace mxfa;

namespace mxfa {

int sm_count_current_device() {
  static std::atomic<int> count[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = count[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  if (dev >= 0 && dev < kMaxDevices) count[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace mxfa

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// u8 tensor [tokens][H][128] as a 3-D map, box 128 x 1 x box_rows, 128B swizzle.
bool make_map_u8(CUtensorMap* m, const void* ptr, int64_t tokens, int H, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, cuuint64_t(H), cuuint64_t(tokens)};
  cuuint64_t strides[2] = {128, cuuint64_t(H) * 128};
  cuuint32_t box[3] = {128, 1, cuuint32_t(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// dQ accumulator [tokens][H][128] (fp32 or fp16) as a 3-D map, box 128 x 1 x 64.
bool make_map_acc(CUtensorMap* m, const void* ptr, int64_t tokens, int H, bool half) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t esz = half ? 2 : 4;
  cuuint64_t dims[3] = {128, cuuint64_t(H), cuuint64_t(tokens)};
  cuuint64_t strides[2] = {128 * esz, cuuint64_t(H) * 128 * esz};
  cuuint32_t box[3] = {128, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor [tokens][H][128] as a 3-D map for stores, box 64 x 1 x 32 (128-byte rows),
// 128B swizzle.
bool make_map_bf16_store(CUtensorMap* m, void* ptr, int64_t tokens, int H) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, cuuint64_t(H), cuuint64_t(tokens)};
  cuuint64_t strides[2] = {256, cuuint64_t(H) * 256};
  cuuint32_t box[3] = {64, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor [tokens][H][128] as a 3-D map for loads, box 128 x heads x 32
// (32 rows of `heads` adjacent heads), no swizzle; rows and heads past the
// tensor read 0.
bool make_map_bf16_rows(CUtensorMap* m, const void* ptr, int64_t tokens, int H, int heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, cuuint64_t(H), cuuint64_t(tokens)};
  cuuint64_t strides[2] = {256, cuuint64_t(H) * 256};
  cuuint32_t box[3] = {128, cuuint32_t(heads), 32};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

mxfa_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MXFA_OK;
  if (e == cudaErrorInvalidValue) return MXFA_ERR_INVALID_ARG;
  return MXFA_ERR_CUDA;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Backward tile records: 2560 bytes per (64-query tile, head); sum over
// sequences of ceil(len / 64) is at most ceil(total / 64) + nseq.
size_t bwd_records_bytes(int64_t total_q, int nseq, int H) {
  const size_t n = size_t(ceil_div(total_q, 64) + nseq) * size_t(H) * 2560u;
  return (n + 255) & ~size_t(255);
}

// Shared checks of a sequence description.
mxfa_status check_seqs(const int32_t* cu, int nseq, int maxlen, int64_t tokens) {
  if (nseq <= 0 || maxlen < 0 || tokens < 0) return MXFA_ERR_INVALID_ARG;
  if (!cu && int64_t(nseq) * maxlen != tokens) return MXFA_ERR_INVALID_ARG;
  if (tokens >= (int64_t(1) << 31)) return MXFA_ERR_UNSUPPORTED;
  return MXFA_OK;
}

mxfa_status check_mx(const mxfa_mx* x) {
  if (!x || !x->data || !x->sf) return MXFA_ERR_INVALID_ARG;
  if (!aligned16(x->data) || !aligned16(x->sf)) return MXFA_ERR_MISALIGNED;
  return MXFA_OK;
}

// Options: NULL = defaults; otherwise checked.
mxfa_status read_opts(const mxfa_attn_opts* opts, float& thr, int& p_scale) {
  thr = MXFA_FWD_RESCALE_THRESHOLD;
  p_scale = MXFA_P_SCALE_BLOCK;
  if (!opts) return MXFA_OK;
  if (!(opts->rescale_threshold >= 0.0f && opts->rescale_threshold <= 8.0f)) return MXFA_ERR_INVALID_ARG;
  if (opts->p_scale != MXFA_P_SCALE_BLOCK && opts->p_scale != MXFA_P_SCALE_CONST) return MXFA_ERR_INVALID_ARG;
  thr = opts->rescale_threshold;
  p_scale = opts->p_scale;
  return MXFA_OK;
}

mxfa_status gemm_common(const mxfa_mx* a, int a_code, const mxfa_mx* b, int b_code, int64_t M, int64_t N,
                        int64_t K, void* y_bf16, const mxfa_mx_out* y_row, const mxfa_mx_out* y_col,
                        mxfa_stream_t stream);

mxfa_status fwd_common(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, Seqs sq, Seqs sk,
                       int64_t total_q, int64_t total_k, int64_t ptq, int64_t ptk, int H, int D,
                       float scale, int causal, void* o, float* lse, const mxfa_mx_out* omx, bool dense,
                       mxfa_stream_t stream, const mxfa_attn_opts* opts = nullptr) {
  mxfa_status s;
  float thr;
  int p_scale;
  if ((s = read_opts(opts, thr, p_scale))) return s;
  if ((s = check_mx(q)) || (s = check_mx(k)) || (s = check_mx(v))) return s;
  if (!o || !lse || H <= 0) return MXFA_ERR_INVALID_ARG;
  if (omx && (!omx->data || !aligned16(omx->data) || (omx->sf_compact && !aligned4(omx->sf_compact)) ||
              (omx->sf_packed && !aligned16(omx->sf_packed))))
    return omx->data ? MXFA_ERR_MISALIGNED : MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return MXFA_ERR_INVALID_ARG;
  if (!aligned16(o)) return MXFA_ERR_MISALIGNED;
  if (ptq <= 0 || ptk <= 0) return MXFA_ERR_INVALID_ARG;
  if (total_q == 0) return MXFA_OK;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_map_u8(&a.tm_q, q->data, total_q, H, 128) || !make_map_u8(&a.tm_k, k->data, total_k, H, 128) ||
      !make_map_u8(&a.tm_v, v->data, total_k, H, 128) || !make_map_bf16_store(&a.tm_o, o, total_q, H))
    return MXFA_ERR_CUDA;
  a.sfq = q->sf;
  a.sfk = k->sf;
  a.sfv = v->sf;
  a.sq = sq;
  a.sk = sk;
  a.total_q = total_q;
  a.ptiles_q = ptq;
  a.ptiles_k = ptk;
  a.H = H;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.rescale_thr = thr;
  // constant P scale: 2^(ceil(thr) - 8), the largest possible P~ = 2^ceil(thr) -> 256
  a.p_sc_const = p_scale == MXFA_P_SCALE_CONST ? uint32_t(127 + int(std::ceil(thr)) - 8) : 0u;
  a.causal = causal ? 1 : 0;
  a.o = static_cast<uint16_t*>(o);
  if (omx) {
    a.omx = omx->data;
    a.omx_sfc = omx->sf_compact;
    a.omx_sfp = omx->sf_packed;
  }
  a.lse = lse;
  a.dense_lse = dense ? 1 : 0;
  a.lse_hstride = dense ? sq.seqlen : total_q;
  // Staged TMA stores of O (and one K/V stage fewer) pay off when items are
  // short, the epilogue being a large share of each item, and cost 1-2% on
  // long ones: mean key length up to 2048.
  a.stage_o = total_k <= int64_t(sk.nseq) * 2048 ? 1 : 0;
  return from_cuda(launch_fwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status bwd_common(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dmx,
                       const void* o, const void* dout, const float* lse, Seqs sq, Seqs sk,
                       int64_t total_q, int64_t total_k, int64_t ptq, int64_t ptk, int H, int D,
                       float scale, int causal, int dq_mode, float dq_static_scale, void* dq, void* dk,
                       void* dv, void* ws, size_t ws_bytes, const mxfa_mx_out* gmx[3], bool dense,
                       mxfa_stream_t stream, const mxfa_attn_opts* opts = nullptr) {
  mxfa_status s;
  float thr_unused;
  int p_scale;
  if ((s = read_opts(opts, thr_unused, p_scale))) return s;
  if ((s = check_mx(q)) || (s = check_mx(k)) || (s = check_mx(v)) || (s = check_mx(dmx))) return s;
  for (int i = 0; i < 3 && gmx; i++) {
    const mxfa_mx_out* m = gmx[i];
    if (!m) continue;
    if (!m->data) return MXFA_ERR_INVALID_ARG;
    if (i == 0 && m->sf_packed && !m->sf_compact) return MXFA_ERR_INVALID_ARG;
    if (!aligned16(m->data) || (m->sf_compact && !aligned4(m->sf_compact)) ||
        (m->sf_packed && !aligned16(m->sf_packed)))
      return MXFA_ERR_MISALIGNED;
  }
  if (!o || !dout || !lse || !dq || !dk || !dv || H <= 0) return MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return MXFA_ERR_INVALID_ARG;
  if (dq_mode != 0 && dq_mode != 1) return MXFA_ERR_INVALID_ARG;
  if (dq_mode == 1) {
    int e;
    if (!(dq_static_scale > 0.0f) || !std::isfinite(dq_static_scale) ||
        std::frexp(dq_static_scale, &e) != 0.5f)
      return MXFA_ERR_INVALID_ARG;  // must be a power of two
  }
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(ws))
    return MXFA_ERR_MISALIGNED;
  if (ptq <= 0 || ptk <= 0) return MXFA_ERR_INVALID_ARG;
  if (!ws) return MXFA_ERR_INVALID_ARG;
  if (ws_bytes < mxfa_bwd_workspace_size(total_q, sq.nseq, H, D, dq_mode))
    return MXFA_ERR_WORKSPACE_TOO_SMALL;
  if (total_q == 0 || total_k == 0) return MXFA_OK;
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_map_u8(&a.tm_q, q->data, total_q, H, 64) || !make_map_u8(&a.tm_do, dmx->data, total_q, H, 64) ||
      !make_map_u8(&a.tm_k, k->data, total_k, H, 128) || !make_map_u8(&a.tm_v, v->data, total_k, H, 128) ||
      !make_map_bf16_store(&a.tm_dk, dk, total_k, H) || !make_map_bf16_store(&a.tm_dv, dv, total_k, H))
    return MXFA_ERR_CUDA;
  a.sfq = q->sf;
  a.sfk = k->sf;
  a.sfv = v->sf;
  a.sfdo = dmx->sf;
  a.do_q = dmx->data;
  a.o = static_cast<const uint16_t*>(o);
  a.dout = static_cast<const uint16_t*>(dout);
  a.lse = lse;
  a.sq = sq;
  a.sk = sk;
  a.total_q = total_q;
  a.total_k = total_k;
  a.ptiles_q = ptq;
  a.ptiles_k = ptk;
  a.H = H;
  a.scale = scale;
  // constant P^T scale 2^-8: P <= 1 maps to <= 256
  a.p_sc_const = p_scale == MXFA_P_SCALE_CONST ? 119u : 0u;
  a.causal = causal ? 1 : 0;
  a.dq_mode = dq_mode;
  a.dq_static_scale = dq_mode == 1 ? dq_static_scale : 1.0f;
  a.dq = static_cast<uint16_t*>(dq);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  if (gmx && gmx[0]) {
    a.dqmx = gmx[0]->data;
    a.dqmx_sfc = gmx[0]->sf_compact;
    a.dqmx_sfp = gmx[0]->sf_packed;
  }
  if (gmx && gmx[1]) {
    a.dkmx = gmx[1]->data;
    a.dkmx_sfc = gmx[1]->sf_compact;
    a.dkmx_sfp = gmx[1]->sf_packed;
  }
  if (gmx && gmx[2]) {
    a.dvmx = gmx[2]->data;
    a.dvmx_sfc = gmx[2]->sf_compact;
    a.dvmx_sfp = gmx[2]->sf_packed;
  }
  a.rec = static_cast<uint8_t*>(ws);
  a.dq_acc = static_cast<uint8_t*>(ws) + bwd_records_bytes(total_q, sq.nseq, H);
  if (!make_map_acc(&a.tm_dqacc, a.dq_acc, total_q, H, dq_mode == 1)) return MXFA_ERR_CUDA;
  a.dense_lse = dense ? 1 : 0;
  a.lse_hstride = dense ? sq.seqlen : total_q;
  return from_cuda(launch_bwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char* mxfa_status_string(mxfa_status s) {
  switch (s) {
    case MXFA_OK: return "ok";
    case MXFA_ERR_INVALID_ARG: return "invalid argument";
    case MXFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MXFA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MXFA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MXFA_ERR_CUDA: return "CUDA error";
    case MXFA_ERR_TIMEOUT: return "device wait timed out";
    case MXFA_ERR_DEVICE_INDEX: return "device index check failed";
  }
  return "unknown status";
}

int mxfa_version(void) { return 1; }

int64_t mxfa_packed_tiles(const int32_t* cu, int nseq, int seqlen) {
  if (nseq < 0) return -1;
  if (!cu) return seqlen < 0 ? -1 : int64_t(nseq) * ceil_div(seqlen, 128);
  int64_t t = 0;
  for (int i = 0; i < nseq; i++) {
    int64_t len = int64_t(cu[i + 1]) - cu[i];
    if (len < 0) return -1;
    t += ceil_div(len, 128);
  }
  return t;
}

size_t mxfa_sf_packed_bytes(mxfa_block blk, int64_t tiles, int H) {
  if (tiles < 0 || H <= 0) return 0;
  return size_t(tiles) * size_t(H) * (blk == MXFA_BLK_SQ ? 16u : 512u);
}

mxfa_status mxfa_quantize(const void* x, int64_t tokens, int H, int D, mxfa_block blk,
                          const int32_t* cu, int nseq, int max_seqlen, int64_t packed_tiles,
                          const mxfa_mx_out* out, mxfa_stream_t stream) {
  if (!x || !out || !out->data || H <= 0) return MXFA_ERR_INVALID_ARG;
  if (blk < MXFA_BLK_ROW || blk > MXFA_BLK_SQ) return MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  mxfa_status s = check_seqs(cu, nseq, max_seqlen, tokens);
  if (s) return s;
  if (!aligned16(x) || !aligned16(out->data)) return MXFA_ERR_MISALIGNED;
  if (out->sf_packed && packed_tiles <= 0) return MXFA_ERR_INVALID_ARG;
  QuantArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const uint16_t*>(x);
  a.tokens = tokens;
  a.H = H;
  a.D = D;
  a.mode = int(blk);
  a.seq = Seqs{cu, nseq, max_seqlen};
  a.packed_tiles = packed_tiles;
  a.data = out->data;
  a.sf_compact = out->sf_compact;
  a.sf_packed = out->sf_packed;
  if (tokens == 0) return MXFA_OK;
  return from_cuda(launch_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status mxfa_quantize_dual(const void* x, int64_t tokens, int H, int D, mxfa_block blk,
                               const int32_t* cu, int nseq, int max_seqlen, int64_t packed_tiles,
                               const mxfa_mx_out* out, const mxfa_mx_out* out_row, mxfa_stream_t stream) {
  if (!x || !out || !out->data || !out_row || !out_row->data || H <= 0) return MXFA_ERR_INVALID_ARG;
  if (blk != MXFA_BLK_COL && blk != MXFA_BLK_SQ) return MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  mxfa_status s = check_seqs(cu, nseq, max_seqlen, tokens);
  if (s) return s;
  if (!aligned16(x) || !aligned16(out->data) || !aligned16(out_row->data)) return MXFA_ERR_MISALIGNED;
  if ((out->sf_packed || out_row->sf_packed) && packed_tiles <= 0) return MXFA_ERR_INVALID_ARG;
  QuantArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const uint16_t*>(x);
  a.tokens = tokens;
  a.H = H;
  a.D = D;
  a.mode = int(blk);
  a.seq = Seqs{cu, nseq, max_seqlen};
  a.packed_tiles = packed_tiles;
  a.data = out->data;
  a.sf_compact = out->sf_compact;
  a.sf_packed = out->sf_packed;
  a.row_data = out_row->data;
  a.row_sfc = out_row->sf_compact;
  a.row_sfp = out_row->sf_packed;
  if (tokens == 0) return MXFA_OK;
  // dense batches of at least one unit's heads take the streaming kernel (its
  // TMA row coordinate is a 32-bit integer)
  a.has_map = (!cu && H >= kQuantHeadsPerUnit && tokens < (int64_t(1) << 31) &&
               make_map_bf16_rows(&a.tm_x, x, tokens, H, kQuantHeadsPerUnit))
                  ? 1
                  : 0;
  return from_cuda(launch_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status mxfa_sf_pack(const uint8_t* sf_compact, int64_t tokens, int H, int D, mxfa_block blk,
                         const int32_t* cu, int nseq, int max_seqlen, int64_t packed_tiles,
                         uint8_t* sf_packed, mxfa_stream_t stream) {
  if (!sf_compact || !sf_packed || H <= 0 || packed_tiles <= 0) return MXFA_ERR_INVALID_ARG;
  if (blk < MXFA_BLK_ROW || blk > MXFA_BLK_SQ) return MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  mxfa_status s = check_seqs(cu, nseq, max_seqlen, tokens);
  if (s) return s;
  PackArgs a;
  a.sf_compact = sf_compact;
  a.tokens = tokens;
  a.H = H;
  a.D = D;
  a.mode = int(blk);
  a.seq = Seqs{cu, nseq, max_seqlen};
  a.packed_tiles = packed_tiles;
  a.sf_packed = sf_packed;
  if (tokens == 0) return MXFA_OK;
  return from_cuda(launch_sf_pack(a, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status mxfa_sf_unpack(const uint8_t* sf_packed, int64_t tokens, int H, int D, mxfa_block blk,
                           const int32_t* cu, int nseq, int max_seqlen, int64_t packed_tiles,
                           uint8_t* sf_compact, mxfa_stream_t stream) {
  if (!sf_compact || !sf_packed || H <= 0 || packed_tiles <= 0) return MXFA_ERR_INVALID_ARG;
  if (blk < MXFA_BLK_ROW || blk > MXFA_BLK_SQ) return MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  mxfa_status s = check_seqs(cu, nseq, max_seqlen, tokens);
  if (s) return s;
  PackArgs a;
  a.sf_compact = nullptr;
  a.tokens = tokens;
  a.H = H;
  a.D = D;
  a.mode = int(blk);
  a.seq = Seqs{cu, nseq, max_seqlen};
  a.packed_tiles = packed_tiles;
  a.sf_packed = const_cast<uint8_t*>(sf_packed);
  if (tokens == 0) return MXFA_OK;
  return from_cuda(launch_sf_unpack(a, sf_compact, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status mxfa_fwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, int B, int S, int H, int D,
                     float softmax_scale, int causal, void* o, float* lse, mxfa_stream_t stream) {
  if (B <= 0 || S <= 0) return MXFA_ERR_INVALID_ARG;
  const int64_t total = int64_t(B) * S;
  mxfa_status s = check_seqs(nullptr, B, S, total);
  if (s) return s;
  const int64_t pt = int64_t(B) * ceil_div(S, 128);
  return fwd_common(q, k, v, Seqs{nullptr, B, S}, Seqs{nullptr, B, S}, total, total, pt, pt, H, D,
                    softmax_scale, causal, o, lse, nullptr, true, stream);
}

mxfa_status mxfa_fwd_mxo(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, int B, int S, int H,
                         int D, float softmax_scale, int causal, void* o, float* lse,
                         const mxfa_mx_out* o_mx, mxfa_stream_t stream) {
  if (B <= 0 || S <= 0 || !o_mx) return MXFA_ERR_INVALID_ARG;
  const int64_t total = int64_t(B) * S;
  mxfa_status s = check_seqs(nullptr, B, S, total);
  if (s) return s;
  const int64_t pt = int64_t(B) * ceil_div(S, 128);
  return fwd_common(q, k, v, Seqs{nullptr, B, S}, Seqs{nullptr, B, S}, total, total, pt, pt, H, D,
                    softmax_scale, causal, o, lse, o_mx, true, stream);
}

mxfa_status mxfa_varlen_fwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const int32_t* cu_q,
                            const int32_t* cu_k, int nseq, int max_sq, int max_sk, int64_t total_q,
                            int64_t total_k, int64_t ptq, int64_t ptk, int H, int D, float softmax_scale,
                            int causal, void* o, float* lse, mxfa_stream_t stream) {
  if (!cu_q || !cu_k) return MXFA_ERR_INVALID_ARG;
  mxfa_status s;
  if ((s = check_seqs(cu_q, nseq, max_sq, total_q)) || (s = check_seqs(cu_k, nseq, max_sk, total_k)))
    return s;
  if (max_sk <= 0) return MXFA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, Seqs{cu_q, nseq, max_sq}, Seqs{cu_k, nseq, max_sk}, total_q, total_k, ptq,
                    ptk, H, D, softmax_scale, causal, o, lse, nullptr, false, stream);
}

mxfa_status mxfa_varlen_fwd_mxo(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                const int32_t* cu_q, const int32_t* cu_k, int nseq, int max_sq,
                                int max_sk, int64_t total_q, int64_t total_k, int64_t ptq, int64_t ptk,
                                int H, int D, float softmax_scale, int causal, void* o, float* lse,
                                const mxfa_mx_out* o_mx, mxfa_stream_t stream) {
  if (!cu_q || !cu_k || !o_mx) return MXFA_ERR_INVALID_ARG;
  mxfa_status s;
  if ((s = check_seqs(cu_q, nseq, max_sq, total_q)) || (s = check_seqs(cu_k, nseq, max_sk, total_k)))
    return s;
  if (max_sk <= 0) return MXFA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, Seqs{cu_q, nseq, max_sq}, Seqs{cu_k, nseq, max_sk}, total_q, total_k, ptq,
                    ptk, H, D, softmax_scale, causal, o, lse, o_mx, false, stream);
}

mxfa_status mxfa_fwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, int B, int S, int H,
                          int D, float softmax_scale, int causal, const mxfa_attn_opts* opts, void* o,
                          float* lse, mxfa_stream_t stream) {
  if (B <= 0 || S <= 0) return MXFA_ERR_INVALID_ARG;
  const int64_t total = int64_t(B) * S;
  mxfa_status s = check_seqs(nullptr, B, S, total);
  if (s) return s;
  const int64_t pt = int64_t(B) * ceil_div(S, 128);
  return fwd_common(q, k, v, Seqs{nullptr, B, S}, Seqs{nullptr, B, S}, total, total, pt, pt, H, D,
                    softmax_scale, causal, o, lse, nullptr, true, stream, opts);
}

mxfa_status mxfa_varlen_fwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                 const int32_t* cu_q, const int32_t* cu_k, int nseq, int max_sq,
                                 int max_sk, int64_t total_q, int64_t total_k, int64_t ptq, int64_t ptk,
                                 int H, int D, float softmax_scale, int causal,
                                 const mxfa_attn_opts* opts, void* o, float* lse, mxfa_stream_t stream) {
  if (!cu_q || !cu_k) return MXFA_ERR_INVALID_ARG;
  mxfa_status s;
  if ((s = check_seqs(cu_q, nseq, max_sq, total_q)) || (s = check_seqs(cu_k, nseq, max_sk, total_k)))
    return s;
  if (max_sk <= 0) return MXFA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, Seqs{cu_q, nseq, max_sq}, Seqs{cu_k, nseq, max_sk}, total_q, total_k, ptq,
                    ptk, H, D, softmax_scale, causal, o, lse, nullptr, false, stream, opts);
}

size_t mxfa_bwd_workspace_size(int64_t total_q, int nseq, int H, int D, int dq_mode) {
  if (total_q < 0 || nseq <= 0 || H <= 0 || D <= 0) return 0;
  return bwd_records_bytes(total_q, nseq, H) + size_t(total_q) * H * D * (dq_mode == 1 ? 2u : 4u);
}

mxfa_status mxfa_bwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dmx,
                     const void* o, const void* dout, const float* lse, int B, int S, int H, int D,
                     float softmax_scale, int causal, int dq_mode, float dq_static_scale, void* dq,
                     void* dk, void* dv, void* ws, size_t ws_bytes, mxfa_stream_t stream) {
  if (B <= 0 || S <= 0) return MXFA_ERR_INVALID_ARG;
  const int64_t total = int64_t(B) * S;
  mxfa_status s = check_seqs(nullptr, B, S, total);
  if (s) return s;
  const int64_t pt = int64_t(B) * ceil_div(S, 128);
  return bwd_common(q, k, v, dmx, o, dout, lse, Seqs{nullptr, B, S}, Seqs{nullptr, B, S}, total, total,
                    pt, pt, H, D, softmax_scale, causal, dq_mode, dq_static_scale, dq, dk, dv, ws,
                    ws_bytes, nullptr, true, stream);
}

mxfa_status mxfa_bwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dmx,
                          const void* o, const void* dout, const float* lse, int B, int S, int H, int D,
                          float softmax_scale, int causal, const mxfa_attn_opts* opts, int dq_mode,
                          float dq_static_scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                          mxfa_stream_t stream) {
  if (B <= 0 || S <= 0) return MXFA_ERR_INVALID_ARG;
  const int64_t total = int64_t(B) * S;
  mxfa_status s = check_seqs(nullptr, B, S, total);
  if (s) return s;
  const int64_t pt = int64_t(B) * ceil_div(S, 128);
  return bwd_common(q, k, v, dmx, o, dout, lse, Seqs{nullptr, B, S}, Seqs{nullptr, B, S}, total, total,
                    pt, pt, H, D, softmax_scale, causal, dq_mode, dq_static_scale, dq, dk, dv, ws,
                    ws_bytes, nullptr, true, stream, opts);
}

mxfa_status mxfa_varlen_bwd_opts(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                 const mxfa_mx* dmx, const void* o, const void* dout, const float* lse,
                                 const int32_t* cu_q, const int32_t* cu_k, int nseq, int max_sq,
                                 int max_sk, int64_t total_q, int64_t total_k, int64_t ptq, int64_t ptk,
                                 int H, int D, float softmax_scale, int causal,
                                 const mxfa_attn_opts* opts, int dq_mode, float dq_static_scale,
                                 void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                                 mxfa_stream_t stream) {
  if (!cu_q || !cu_k) return MXFA_ERR_INVALID_ARG;
  mxfa_status s;
  if ((s = check_seqs(cu_q, nseq, max_sq, total_q)) || (s = check_seqs(cu_k, nseq, max_sk, total_k)))
    return s;
  return bwd_common(q, k, v, dmx, o, dout, lse, Seqs{cu_q, nseq, max_sq}, Seqs{cu_k, nseq, max_sk},
                    total_q, total_k, ptq, ptk, H, D, softmax_scale, causal, dq_mode, dq_static_scale,
                    dq, dk, dv, ws, ws_bytes, nullptr, false, stream, opts);
}

mxfa_status mxfa_bwd_mxg(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dmx,
                         const void* o, const void* dout, const float* lse, int B, int S, int H, int D,
                         float softmax_scale, int causal, int dq_mode, float dq_static_scale, void* dq,
                         void* dk, void* dv, void* ws, size_t ws_bytes, const mxfa_mx_out* dq_mx,
                         const mxfa_mx_out* dk_mx, const mxfa_mx_out* dv_mx, mxfa_stream_t stream) {
  if (B <= 0 || S <= 0) return MXFA_ERR_INVALID_ARG;
  const int64_t total = int64_t(B) * S;
  mxfa_status s = check_seqs(nullptr, B, S, total);
  if (s) return s;
  const int64_t pt = int64_t(B) * ceil_div(S, 128);
  const mxfa_mx_out* gmx[3] = {dq_mx, dk_mx, dv_mx};
  return bwd_common(q, k, v, dmx, o, dout, lse, Seqs{nullptr, B, S}, Seqs{nullptr, B, S}, total, total,
                    pt, pt, H, D, softmax_scale, causal, dq_mode, dq_static_scale, dq, dk, dv, ws,
                    ws_bytes, gmx, true, stream);
}

mxfa_status mxfa_varlen_bwd(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dmx,
                            const void* o, const void* dout, const float* lse, const int32_t* cu_q,
                            const int32_t* cu_k, int nseq, int max_sq, int max_sk, int64_t total_q,
                            int64_t total_k, int64_t ptq, int64_t ptk, int H, int D, float softmax_scale,
                            int causal, int dq_mode, float dq_static_scale, void* dq, void* dk, void* dv,
                            void* ws, size_t ws_bytes, mxfa_stream_t stream) {
  if (!cu_q || !cu_k) return MXFA_ERR_INVALID_ARG;
  mxfa_status s;
  if ((s = check_seqs(cu_q, nseq, max_sq, total_q)) || (s = check_seqs(cu_k, nseq, max_sk, total_k)))
    return s;
  return bwd_common(q, k, v, dmx, o, dout, lse, Seqs{cu_q, nseq, max_sq}, Seqs{cu_k, nseq, max_sk},
                    total_q, total_k, ptq, ptk, H, D, softmax_scale, causal, dq_mode, dq_static_scale,
                    dq, dk, dv, ws, ws_bytes, nullptr, false, stream);
}

mxfa_status mxfa_varlen_bwd_mxg(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v, const mxfa_mx* dmx,
                                const void* o, const void* dout, const float* lse, const int32_t* cu_q,
                                const int32_t* cu_k, int nseq, int max_sq, int max_sk, int64_t total_q,
                                int64_t total_k, int64_t ptq, int64_t ptk, int H, int D,
                                float softmax_scale, int causal, int dq_mode, float dq_static_scale,
                                void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                                const mxfa_mx_out* dq_mx, const mxfa_mx_out* dk_mx,
                                const mxfa_mx_out* dv_mx, mxfa_stream_t stream) {
  if (!cu_q || !cu_k) return MXFA_ERR_INVALID_ARG;
  mxfa_status s;
  if ((s = check_seqs(cu_q, nseq, max_sq, total_q)) || (s = check_seqs(cu_k, nseq, max_sk, total_k)))
    return s;
  const mxfa_mx_out* gmx[3] = {dq_mx, dk_mx, dv_mx};
  return bwd_common(q, k, v, dmx, o, dout, lse, Seqs{cu_q, nseq, max_sq}, Seqs{cu_k, nseq, max_sk},
                    total_q, total_k, ptq, ptk, H, D, softmax_scale, causal, dq_mode, dq_static_scale,
                    dq, dk, dv, ws, ws_bytes, gmx, false, stream);
}

mxfa_status mxfa_rmsnorm_quant(const void* x, const float* gamma, int64_t T, int64_t C, float eps,
                               int seg_len, int H, const mxfa_mx_out* row, const mxfa_mx_out* col,
                               const mxfa_mx_out* sq, mxfa_stream_t stream) {
  if (!x || !gamma || T < 0 || seg_len <= 0 || H <= 0) return MXFA_ERR_INVALID_ARG;
  if (!row && !col && !sq) return MXFA_ERR_INVALID_ARG;
  if (C != 256 && C != 512 && C != 1024 && C != 2048) return MXFA_ERR_UNSUPPORTED;
  if (C % H != 0 || C / H != 128) return MXFA_ERR_UNSUPPORTED;
  if (seg_len % 32 != 0) return MXFA_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return MXFA_ERR_INVALID_ARG;
  const mxfa_mx_out* outs[3] = {row, col, sq};
  bool packed = false;
  for (const mxfa_mx_out* m : outs) {
    if (!m) continue;
    if (!m->data) return MXFA_ERR_INVALID_ARG;
    if (!aligned16(m->data)) return MXFA_ERR_MISALIGNED;
    if (m->sf_packed) packed = true;
  }
  if (packed && (seg_len % 128 != 0 || T % seg_len != 0)) return MXFA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(gamma)) return MXFA_ERR_MISALIGNED;
  RmsArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const uint16_t*>(x);
  a.gamma = gamma;
  a.T = T;
  a.C = int(C);
  a.eps = eps;
  a.seg_len = seg_len;
  a.H = H;
  a.D = 128;
  if (row) { a.row_data = row->data; a.row_sfc = row->sf_compact; a.row_sfp = row->sf_packed; }
  if (col) { a.col_data = col->data; a.col_sfc = col->sf_compact; a.col_sfp = col->sf_packed; }
  if (sq) { a.sq_data = sq->data; a.sq_sfc = sq->sf_compact; a.sq_sfp = sq->sf_packed; }
  if (T == 0) return MXFA_OK;
  return from_cuda(launch_rmsnorm_quant(a, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status mxfa_gemm_quant_fmt(const mxfa_mx* a, int a_fmt, const mxfa_mx* b, int b_fmt, int64_t M,
                                int64_t N, int64_t K, void* y_bf16, const mxfa_mx_out* y_row,
                                const mxfa_mx_out* y_col, mxfa_stream_t stream) {
  // element formats -> the MMA kind's format codes
  auto code = [](int f) { return f == MXFA_ELEM_E4M3 ? 0 : f == MXFA_ELEM_E2M3 ? 3 : f == MXFA_ELEM_E3M2 ? 4 : 5; };
  for (int f : {a_fmt, b_fmt})
    if (f != MXFA_ELEM_E4M3 && f != MXFA_ELEM_E2M3 && f != MXFA_ELEM_E3M2 && f != MXFA_ELEM_E2M1)
      return MXFA_ERR_INVALID_ARG;
  return gemm_common(a, code(a_fmt), b, code(b_fmt), M, N, K, y_bf16, y_row, y_col, stream);
}

mxfa_status mxfa_gemm_quant(const mxfa_mx* a, const mxfa_mx* b, int64_t M, int64_t N, int64_t K,
                            void* y_bf16, const mxfa_mx_out* y_row, const mxfa_mx_out* y_col,
                            mxfa_stream_t stream) {
  return gemm_common(a, 0, b, 0, M, N, K, y_bf16, y_row, y_col, stream);
}

mxfa_status mxfa_quantize_lowp(const void* x, int64_t rows, int cols, int fmt, int q_layout, uint8_t* q,
                               uint8_t* sf, uint8_t* sf_packed, float* tensor_scale, mxfa_stream_t stream) {
  if (!x || !q || !sf || rows < 0 || cols <= 0) return MXFA_ERR_INVALID_ARG;
  if (fmt < MXFA_LOWP_MXFP4 || fmt > MXFA_LOWP_NVFP4) return MXFA_ERR_INVALID_ARG;
  if (q_layout != MXFA_LOWP_CODES && q_layout != MXFA_LOWP_MMA) return MXFA_ERR_INVALID_ARG;
  if (q_layout == MXFA_LOWP_MMA && fmt == MXFA_LOWP_NVFP4) return MXFA_ERR_UNSUPPORTED;
  if (cols % (fmt == MXFA_LOWP_NVFP4 ? 16 : 32) != 0) return MXFA_ERR_UNSUPPORTED;
  if (fmt == MXFA_LOWP_NVFP4 && (!tensor_scale || !aligned4(tensor_scale))) return MXFA_ERR_INVALID_ARG;
  if (sf_packed && (fmt == MXFA_LOWP_NVFP4 || rows % 128 != 0 || cols % 128 != 0)) return MXFA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(q) || (sf_packed && !aligned16(sf_packed))) return MXFA_ERR_MISALIGNED;
  if (rows * int64_t(cols) >= (int64_t(1) << 40)) return MXFA_ERR_UNSUPPORTED;
  LowpArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.fmt = fmt;
  a.q = q;
  a.q_mma = q_layout == MXFA_LOWP_MMA;
  a.sf = sf;
  a.sf_packed = sf_packed;
  a.tensor_scale = tensor_scale;
  return from_cuda(launch_lowp_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
mxfa_status gemm_common(const mxfa_mx* a, int a_code, const mxfa_mx* b, int b_code, int64_t M, int64_t N,
                        int64_t K, void* y_bf16, const mxfa_mx_out* y_row, const mxfa_mx_out* y_col,
                        mxfa_stream_t stream) {
  mxfa_status s;
  if ((s = check_mx(a)) || (s = check_mx(b))) return s;
  if (M < 0 || N < 0 || K < 0) return MXFA_ERR_INVALID_ARG;
  if (M % 128 || N % 128 || K % 128) return MXFA_ERR_UNSUPPORTED;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 24) || K >= (int64_t(1) << 24)) return MXFA_ERR_UNSUPPORTED;
  if (!y_bf16 && !y_row && !y_col) return MXFA_ERR_INVALID_ARG;
  if (y_bf16 && !aligned16(y_bf16)) return MXFA_ERR_MISALIGNED;
  for (const mxfa_mx_out* m : {y_row, y_col}) {
    if (!m) continue;
    if (!m->data) return MXFA_ERR_INVALID_ARG;
    if (!aligned16(m->data) || (m->sf_compact && !aligned4(m->sf_compact)) ||
        (m->sf_packed && !aligned16(m->sf_packed)))
      return MXFA_ERR_MISALIGNED;
  }
  if (M == 0 || N == 0) return MXFA_OK;
  if (K == 0) return MXFA_ERR_UNSUPPORTED;
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  if (!make_map_u8(&g.tm_a, a->data, M, int(K / 128), 128) || !make_map_u8(&g.tm_b, b->data, N, int(K / 128), 128))
    return MXFA_ERR_CUDA;
  g.sfa = a->sf;
  g.sfb = b->sf;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_fmt = a_code;
  g.b_fmt = b_code;
  g.y_bf16 = static_cast<uint16_t*>(y_bf16);
  if (y_row) { g.row_data = y_row->data; g.row_sfc = y_row->sf_compact; g.row_sfp = y_row->sf_packed; }
  if (y_col) { g.col_data = y_col->data; g.col_sfc = y_col->sf_compact; g.col_sfp = y_col->sf_packed; }
  return from_cuda(launch_gemm_quant(g, reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

mxfa_status mxfa_tensor_peak_probe(int iters, int ctas, unsigned long long* cycles, mxfa_stream_t stream) {
  if (iters <= 0 || ctas <= 0 || !cycles) return MXFA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cycles) & 7u) return MXFA_ERR_MISALIGNED;
  return from_cuda(launch_mma_peak(iters, ctas, cycles, reinterpret_cast<cudaStream_t>(stream)));
}

mxfa_status mxfa_get_device_status(mxfa_stream_t stream, unsigned* flags) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MXFA_ERR_CUDA;
  unsigned f = read_status_quant(st) | read_status_fwd(st) | read_status_bwd(st) | read_status_gemm(st);
  if (flags) *flags = f;
  if (f & 1u) return MXFA_ERR_TIMEOUT;
  if (f & 2u) return MXFA_ERR_DEVICE_INDEX;
  return MXFA_OK;
}

}  // extern "C"
