// api.cu -- the C ABI declared in include/attn_core.h: argument checks,
// TMA tensor-map encoding and kernel launches.  No device memory is
// allocated here; the caller owns every buffer.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include "../../include/attn_core.h"
#include "kernels.h"
#include "philox.cuh"
#include "tile.cuh"

namespace {

using ac::kBlockRows;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder()
{
    if (g_encode) return ATTN_CORE_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return ATTN_CORE_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return ATTN_CORE_OK;
}

// 0: not checked yet, 1: sm_103, -1: other.
int g_dev_ok[128];

int check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_CORE_ERR_CUDA;
    if (dev < 0 || dev >= 128) return ATTN_CORE_ERR_UNSUPPORTED;
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return ATTN_CORE_ERR_CUDA;
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_dev_ok[dev] == 1 ? ATTN_CORE_OK : ATTN_CORE_ERR_UNSUPPORTED;
}

int g_dev_sms[128];

int device_sms(int* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return ATTN_CORE_ERR_CUDA;
    if (g_dev_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return ATTN_CORE_ERR_CUDA;
        g_dev_sms[dev] = n;
    }
    *out = g_dev_sms[dev];
    return ATTN_CORE_OK;
}

bool supported_d(int d) { return d == 64 || d == 96 || d == 128 || d == 160; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Keys per KV head: s_kv, or s when s_kv is 0.
int keys_of(const attn_core_params* p) { return p->s_kv ? p->s_kv : p->s; }

int check_params(const attn_core_params* p)
{
    if (p == nullptr) return ATTN_CORE_ERR_INVALID_ARG;
    if (p->b <= 0 || p->h_q <= 0 || p->h_kv <= 0 || p->s <= 0 || p->d <= 0 || p->s_kv < 0)
        return ATTN_CORE_ERR_INVALID_ARG;
    if (p->h_q % p->h_kv != 0) return ATTN_CORE_ERR_INVALID_ARG;
    if (p->causal != 0 && p->causal != 1) return ATTN_CORE_ERR_INVALID_ARG;
    if (!(p->p_drop >= 0.0f && p->p_drop < 1.0f)) return ATTN_CORE_ERR_INVALID_ARG;
    if (p->offset >> 32) return ATTN_CORE_ERR_INVALID_ARG;
    if (isnan(p->scale) || isinf(p->scale)) return ATTN_CORE_ERR_INVALID_ARG;
    // Counter words and grid sizes are 32-bit.
    const int64_t n_bh = (int64_t)p->b * p->h_q;
    const int64_t n_blk = ((int64_t)p->s + kBlockRows - 1) / kBlockRows;
    const int64_t n_blk_k = ((int64_t)keys_of(p) + kBlockRows - 1) / kBlockRows;
    if (n_bh * n_blk >= (int64_t)INT32_MAX || n_bh * n_blk_k >= (int64_t)INT32_MAX ||
        (int64_t)p->s * n_bh >= ((int64_t)1 << 40))
        return ATTN_CORE_ERR_INVALID_ARG;
    return ATTN_CORE_OK;
}

// Dropout threshold of the attention core on an 8-bit draw: round(p * 256), at
// most 255; an element is dropped iff its draw is below it.
uint32_t drop_threshold(float p)
{
    if (!(p > 0.0f)) return 0u;
    long long t = llround((double)p * 256.0);
    if (t > 255) t = 255;
    if (t < 0) t = 0;
    return (uint32_t)t;
}

// The dropout + layer norm block's threshold on a 16-bit draw: round(p * 65536),
// at most 65535.
uint32_t drop_threshold16(float p)
{
    if (!(p > 0.0f)) return 0u;
    long long t = llround((double)p * 65536.0);
    if (t > 65535) t = 65535;
    if (t < 0) t = 0;
    return (uint32_t)t;
}

ac::CommonArgs common_args(const attn_core_params* p)
{
    ac::CommonArgs c{};
    c.s = p->s;
    c.s_k = keys_of(p);
    c.h_q = p->h_q;
    c.h_kv = p->h_kv;
    c.n_blk = (p->s + kBlockRows - 1) / kBlockRows;
    c.n_blk_k = (c.s_k + kBlockRows - 1) / kBlockRows;
    c.n_bh = p->b * p->h_q;
    c.causal = p->causal;
    const float scale = (p->scale > 0.0f) ? p->scale : 1.0f / sqrtf((float)p->d);
    c.scale = scale;
    c.scale_log2 = scale * 1.44269504088896340736f;
    c.thr = drop_threshold(p->p_drop);
    c.keep_scale = 1.0f / (1.0f - (float)c.thr / 256.0f);
    c.seed_lo = (uint32_t)(p->seed & 0xffffffffu);
    c.seed_hi = (uint32_t)(p->seed >> 32);
    ac::philox_round_keys(c.seed_lo, c.seed_hi, c.rk);
    c.offset = (uint32_t)p->offset;
    c.status = p->dev_status;
    c.timeout_ns = (uint64_t)(p->wait_timeout_ms ? p->wait_timeout_ms : 2000u) * 1000000ull;
    c.inject_timeout = (p->flags & ATTN_CORE_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
    c.bh0 = 0;
    c.lse_stride = p->s;
    return c;
}

// 3-D map over `heads` x `s` rows of d bf16 values, row r of head h at
// ptr + h * head_stride + r * row_stride elements: box = one column chunk of
// `rows` rows of one head, swizzled to match the shared-memory tile layout.
// [heads, s, d] tensors have row_stride d and head_stride s * d; one sequence
// of a packed [tokens, heads, d] batch has row_stride heads * d and
// head_stride d.
int encode_map_strided(CUtensorMap* m, const void* ptr, int d, int s, int64_t heads, int64_t row_stride,
                       int64_t head_stride, int rows)
{
    const int cw = (d % 64 == 0) ? 64 : 32;
    const CUtensorMapSwizzle sw = (cw == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)s, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)head_stride * 2};
    cuuint32_t box[3] = {(cuuint32_t)cw, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_CORE_OK : ATTN_CORE_ERR_CUDA;
}

// Where the query-side (Q, O, dO, dQ) and key-side (K, V, dK, dV) rows of one
// launch live, and where its LSE rows go.
struct Geometry {
    int64_t q_heads, kv_heads;              // map heads: b * h_q and b * h_kv, or h_q and h_kv
    int64_t q_row, q_head, kv_row, kv_head; // strides in elements
    int64_t lse_stride;                     // LSE elements from one query head to the next
    uint32_t bh0;                           // Philox head-index offset
    int64_t q_rows, k_rows;                 // rows per map head: s and s_kv, or a packed
                                            // batch's total query and key counts
    int64_t ws_stride;                      // backward workspace rows per query head
    const int32_t* cu_q;                    // a packed batch's device sequence tables,
    const int32_t* cu_k;                    // or null
};

Geometry padded_geometry(const attn_core_params* p, int sk)
{
    Geometry g;
    g.q_heads = (int64_t)p->b * p->h_q;
    g.kv_heads = (int64_t)p->b * p->h_kv;
    g.q_row = g.kv_row = p->d;
    g.q_head = (int64_t)p->s * p->d;
    g.kv_head = (int64_t)sk * p->d;
    g.lse_stride = p->s;
    g.bh0 = 0;
    g.q_rows = p->s;
    g.k_rows = sk;
    g.ws_stride = ((int64_t)p->s + kBlockRows - 1) / kBlockRows * kBlockRows;
    g.cu_q = g.cu_k = nullptr;
    return g;
}

size_t padded_rows(const attn_core_params* p)
{
    const size_t n_blk = ((size_t)p->s + kBlockRows - 1) / kBlockRows;
    return (size_t)p->b * p->h_q * n_blk * kBlockRows;
}

// Bytes of the keep bits the dQ kernel hands to the dK/dV kernel (p > 0,
// d <= 128).  For d = 160 the dK/dV kernel is bound by its products, not by
// its row threads, so drawing the mask there again costs no time, while
// writing the bits would cost the dQ kernel some: that case draws twice.
size_t mask_bytes(const attn_core_params* p)
{
    if (drop_threshold(p->p_drop) == 0 || p->d > 128 || (p->flags & ATTN_CORE_FLAG_REDRAW_MASK)) return 0;
    // the hand-over layout covers the square causal pattern; causal
    // cross-attention draws the mask twice
    if (p->causal && keys_of(p) != p->s) return 0;
    const ac::CommonArgs c = common_args(p);
    return sizeof(uint32_t) * ac::mask_ws_words(c);
}

int record(void** ev, int idx, cudaStream_t st)
{
    if (!ev) return ATTN_CORE_OK;
    return cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[idx]), st) == cudaSuccess ? ATTN_CORE_OK
                                                                                       : ATTN_CORE_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* attn_core_strerror(int code)
{
    switch (code & 0xff) {
        case ATTN_CORE_OK: return "ok";
        case ATTN_CORE_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_CORE_ERR_UNSUPPORTED: return "unsupported head dimension or device";
        case ATTN_CORE_ERR_MISALIGNED: return "pointer not aligned (16 bytes; workspace 256 bytes)";
        case ATTN_CORE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case ATTN_CORE_ERR_CUDA: return "CUDA error";
        case ATTN_CORE_ERR_DEVICE_TIMEOUT: return "a kernel wait ran past its time limit";
        default: return "unknown error";
    }
}

int attn_core_stored_bytes(const attn_core_params* p, attn_core_bytes* out)
{
    int rc = check_params(p);
    if (rc) return rc;
    if (!out) return ATTN_CORE_ERR_INVALID_ARG;
    const int64_t s = p->s, sk = keys_of(p), b = p->b, a = p->h_q, akv = p->h_kv, d = p->d;
    const int64_t h = a * d;
    out->layer_selective = 34 * s * b * h;
    out->layer_none = out->layer_selective + 5 * a * s * s * b;
    out->layer_full = 2 * s * b * h;
    out->core_scores_avoided = 5 * a * s * sk * b;
    out->core_kept = 2 * d * b * (2 * a * s + 2 * akv * sk);
    out->core_recompute_state = 4 * b * a * s + 16;
    return ATTN_CORE_OK;
}

size_t attn_core_bwd_workspace_bytes(const attn_core_params* p)
{
    if (check_params(p)) return 0;
    return 2 * sizeof(float) * padded_rows(p) + mask_bytes(p);
}

}  // extern "C"

namespace {

// One forward launch over the geometry g (pointers at the launch's first row).
int fwd_launch(const attn_core_params* p, const Geometry& g, const void* q, const void* k, const void* v, void* o,
               float* lse, cudaStream_t st)
{
    int rc;
    const int sk = keys_of(p);
    (void)sk;
    CUtensorMap tq, tk, tv, to;
    if ((rc = encode_map_strided(&tq, q, p->d, (int)g.q_rows, g.q_heads, g.q_row, g.q_head, 128)) ||
        (rc = encode_map_strided(&tk, k, p->d, (int)g.k_rows, g.kv_heads, g.kv_row, g.kv_head, 128)) ||
        (rc = encode_map_strided(&tv, v, p->d, (int)g.k_rows, g.kv_heads, g.kv_row, g.kv_head, 128)) ||
        (rc = encode_map_strided(&to, o, p->d, (int)g.q_rows, g.q_heads, g.q_row, g.q_head, 128)))
        return rc;
    ac::FwdArgs a{};
    a.c = common_args(p);
    a.c.bh0 = g.bh0;
    a.c.lse_stride = g.lse_stride;
    a.c.cu_q = g.cu_q;
    a.c.cu_k = g.cu_k;
    a.c.ws_stride = g.ws_stride;
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.o_head_stride = g.q_head;
    a.o_row_stride = g.q_row;
    if ((rc = device_sms(&a.num_sms))) return rc;
    if ((rc = record(p->timing_events, 0, st))) return rc;
    if (ac::launch_fwd(p->d, a.c.thr != 0, tq, tk, tv, to, a, st) != 0) return ATTN_CORE_ERR_CUDA;
    return record(p->timing_events, 1, st);
}

}  // namespace

extern "C" {

int attn_core_fwd(const attn_core_params* p, const void* q, const void* k, const void* v, void* o, float* lse,
                  void* stream)
{
    int rc = check_params(p);
    if (rc) return rc;
    if (!q || !k || !v || !o || !lse) return ATTN_CORE_ERR_INVALID_ARG;
    if (!supported_d(p->d)) return ATTN_CORE_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_CORE_ERR_MISALIGNED;
    if ((rc = check_device())) return rc;
    if ((rc = get_encoder())) return rc;
    return fwd_launch(p, padded_geometry(p, keys_of(p)), q, k, v, o, lse, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Workspace bytes of one backward launch: the two row statistics and (when
// shared) the keep bits, rounded up to 256 bytes.
size_t launch_ws_bytes(const attn_core_params* p, bool share_mask)
{
    const size_t b = 2 * sizeof(float) * padded_rows(p) + (share_mask ? mask_bytes(p) : 0);
    return (b + 255) & ~(size_t)255;
}

// One backward launch (dQ, then dK/dV) over the geometry g; `workspace` holds
// launch_ws_bytes(p, share_mask) bytes.  share_mask: the workspace also holds
// the keep bits, which the dQ kernel writes and the dK/dV kernel reads;
// otherwise the dK/dV kernel draws the mask again from Philox.
int bwd_launch(const attn_core_params* p, const Geometry& g, const void* q, const void* k, const void* v,
               const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
               bool share_mask, cudaStream_t st)
{
    int rc;
    const int bq = ac::dkdv_query_tile(p->d);
    const int bn = ac::dq_key_tile(p->d);
    const int sk = keys_of(p);
    auto qmap = [&](CUtensorMap* m, const void* ptr, int rows) {
        return encode_map_strided(m, ptr, p->d, (int)g.q_rows, g.q_heads, g.q_row, g.q_head, rows);
    };
    auto kmap = [&](CUtensorMap* m, const void* ptr, int rows) {
        return encode_map_strided(m, ptr, p->d, (int)g.k_rows, g.kv_heads, g.kv_row, g.kv_head, rows);
    };
    CUtensorMap tq128, tdo128, to128, tdq128, tqb, tdob, tk, tv, tkb, tvb, tdk, tdv;
    if ((rc = qmap(&tq128, q, 128)) || (rc = qmap(&tdo128, dout, 128)) || (rc = qmap(&to128, o, 128)) ||
        (rc = qmap(&tdq128, dq, 128)) ||
        (rc = qmap(&tqb, q, bq)) || (rc = qmap(&tdob, dout, bq)) || (rc = kmap(&tk, k, 128)) ||
        (rc = kmap(&tv, v, 128)) || (rc = kmap(&tkb, k, bn)) || (rc = kmap(&tvb, v, bn)) ||
        (rc = kmap(&tdk, dk, 128)) || (rc = kmap(&tdv, dv, 128)))
        return rc;
    ac::BwdArgs a{};
    a.c = common_args(p);
    a.c.bh0 = g.bh0;
    a.c.lse_stride = g.lse_stride;
    a.c.cu_q = g.cu_q;
    a.c.cu_k = g.cu_k;
    a.c.ws_stride = g.ws_stride;
    a.s_pad = a.c.n_blk * kBlockRows;
    const size_t ws_rows = (size_t)g.q_heads * (size_t)g.ws_stride;
    a.o = static_cast<const uint16_t*>(o);
    a.dout = static_cast<const uint16_t*>(dout);
    a.lse = lse;
    a.lse2_ws = static_cast<float*>(workspace);
    a.delta_ws = static_cast<float*>(workspace) + ws_rows;
    a.mask_ws = (share_mask && g.cu_q == nullptr && mask_bytes(p) != 0)
                    ? reinterpret_cast<uint32_t*>(static_cast<float*>(workspace) + 2 * ws_rows)
                    : nullptr;
    a.dq = static_cast<uint16_t*>(dq);
    a.dk = static_cast<uint16_t*>(dk);
    a.dv = static_cast<uint16_t*>(dv);
    a.q_head_stride = g.q_head;
    a.q_row_stride = g.q_row;
    a.kv_head_stride = g.kv_head;
    a.kv_row_stride = g.kv_row;
    a.d = p->d;
    if ((rc = device_sms(&a.num_sms))) return rc;
    const bool drop = a.c.thr != 0;
    if ((rc = record(p->timing_events, 0, st))) return rc;
    if (ac::launch_bwd_dq(p->d, drop, tq128, tkb, tvb, tdo128, to128, tdq128, a, st) != 0) return ATTN_CORE_ERR_CUDA;
    if ((rc = record(p->timing_events, 1, st)) || (rc = record(p->timing_events, 2, st))) return rc;
    if (ac::launch_bwd_dkdv(p->d, drop, tqb, tk, tv, tdob, tdk, tdv, a, st) != 0) return ATTN_CORE_ERR_CUDA;
    // Causal with more keys than queries: keys from the end of the last query
    // block on are seen by no query (top-left alignment) and the dK/dV kernel
    // skips their blocks, so their gradients are set to zero here.
    const int64_t kz = (int64_t)a.c.n_blk * kBlockRows;
    if (g.cu_q == nullptr && p->causal && sk > kz) {
        const size_t row_bytes = (size_t)g.kv_row * sizeof(uint16_t);
        for (void* t : {dk, dv}) {
            uint8_t* base = static_cast<uint8_t*>(t) + (size_t)kz * row_bytes;
            cudaError_t e;
            if (g.kv_head == p->d) {        // token-major rows: all heads of a row are adjacent
                e = cudaMemsetAsync(base, 0, (size_t)(sk - kz) * row_bytes, st);
            } else {                        // head-major: rows kz .. sk - 1 of every head
                e = cudaMemset2DAsync(base, (size_t)g.kv_head * sizeof(uint16_t), 0, (size_t)(sk - kz) * row_bytes,
                                      (size_t)g.kv_heads, st);
            }
            if (e != cudaSuccess) return ATTN_CORE_ERR_CUDA;
        }
    }
    return record(p->timing_events, 3, st);
}

// The backward of the padded layout.
int bwd_impl(const attn_core_params* p, const void* q, const void* k, const void* v, const void* o,
             const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, bool share_mask, void* stream)
{
    int rc = check_params(p);
    if (rc) return rc;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return ATTN_CORE_ERR_INVALID_ARG;
    if (!supported_d(p->d)) return ATTN_CORE_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return ATTN_CORE_ERR_MISALIGNED;
    const size_t need = 2 * sizeof(float) * padded_rows(p) + (share_mask ? mask_bytes(p) : 0);
    if (workspace_bytes < need) return ATTN_CORE_ERR_WORKSPACE_TOO_SMALL;
    if ((rc = check_device())) return rc;
    if ((rc = get_encoder())) return rc;
    return bwd_launch(p, padded_geometry(p, keys_of(p)), q, k, v, o, lse, dout, dq, dk, dv, workspace, share_mask,
                      reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int attn_core_bwd_recompute(const attn_core_params* p, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, void* stream)
{
    return bwd_impl(p, q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, true, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Variable-length (packed) batches: one launch per kernel over the whole batch.
// The kernels take the n_seq sequences as a batch of n_seq elements of the
// longest sequence's length and read each tile's own lengths and first rows
// from the device copies of the sequence tables.
namespace {

struct VarlenShape {
    int64_t total_q, total_k;
    int32_t max_q, max_k;
    const int32_t* cu_q_dev;
    const int32_t* cu_k_dev;
};

// Checks the host sequence tables and the device copies' presence.
int check_varlen(const attn_core_varlen_params* vp, VarlenShape* out)
{
    if (vp == nullptr || vp->n_seq <= 0 || vp->cu_seqlens_q == nullptr) return ATTN_CORE_ERR_INVALID_ARG;
    if (vp->cu_seqlens_q_dev == nullptr || (vp->cu_seqlens_k != nullptr && vp->cu_seqlens_k_dev == nullptr))
        return ATTN_CORE_ERR_INVALID_ARG;
    if (vp->base.timing_events != nullptr) return ATTN_CORE_ERR_INVALID_ARG;
    if ((int64_t)vp->n_seq * vp->base.h_q >= (int64_t)INT32_MAX) return ATTN_CORE_ERR_INVALID_ARG;
    const int32_t* cq = vp->cu_seqlens_q;
    const int32_t* ck = vp->cu_seqlens_k ? vp->cu_seqlens_k : cq;
    if (cq[0] != 0 || ck[0] != 0) return ATTN_CORE_ERR_INVALID_ARG;
    int32_t max_q = 0, max_k = 0;
    for (int i = 0; i < vp->n_seq; ++i) {
        const int32_t lq = cq[i + 1] - cq[i], lk = ck[i + 1] - ck[i];
        if (lq < 0 || lk < 0 || (lq > 0 && lk == 0)) return ATTN_CORE_ERR_INVALID_ARG;
        if (lq > max_q) max_q = lq;
        if (lk > max_k) max_k = lk;
    }
    out->total_q = cq[vp->n_seq];
    out->total_k = ck[vp->n_seq];
    if (out->total_q >= (int64_t)INT32_MAX - 132 * (int64_t)vp->n_seq - 4 || out->total_k >= (int64_t)INT32_MAX)
        return ATTN_CORE_ERR_INVALID_ARG;
    out->max_q = max_q;
    out->max_k = max_k;
    out->cu_q_dev = vp->cu_seqlens_q_dev;
    out->cu_k_dev = vp->cu_seqlens_k ? vp->cu_seqlens_k_dev : vp->cu_seqlens_q_dev;
    return ATTN_CORE_OK;
}

// The batch as one launch: n_seq elements of the longest sequence's length.
attn_core_params batch_params(const attn_core_varlen_params* vp, const VarlenShape& vs)
{
    attn_core_params ps = vp->base;
    ps.b = vp->n_seq;
    ps.s = vs.max_q;
    ps.s_kv = vs.max_k;
    return ps;
}

// Packed [tokens, heads, d] tensors: one map head per attention head, rows of
// the whole batch.
Geometry packed_geometry(const attn_core_varlen_params* vp, const VarlenShape& vs)
{
    Geometry g;
    g.q_heads = vp->base.h_q;
    g.kv_heads = vp->base.h_kv;
    g.q_row = (int64_t)vp->base.h_q * vp->base.d;
    g.kv_row = (int64_t)vp->base.h_kv * vp->base.d;
    g.q_head = g.kv_head = vp->base.d;
    g.lse_stride = vs.total_q;
    g.bh0 = 0;
    g.q_rows = vs.total_q;
    g.k_rows = vs.total_k;
    g.ws_stride = ((vs.total_q + 3) & ~(int64_t)3) + 132 * (int64_t)vp->n_seq;   // see packed_ws_row0
    g.cu_q = vs.cu_q_dev;
    g.cu_k = vs.cu_k_dev;
    return g;
}

size_t varlen_ws_bytes(const attn_core_varlen_params* vp, const VarlenShape& vs)
{
    const size_t rows = (size_t)((vs.total_q + 3) & ~(int64_t)3) + 132 * (size_t)vp->n_seq;
    const size_t b = 2 * sizeof(float) * (size_t)vp->base.h_q * rows;
    return (b + 255) & ~(size_t)255;
}

}  // namespace

extern "C" {

size_t attn_core_bwd_varlen_workspace_bytes(const attn_core_varlen_params* vp)
{
    VarlenShape vs;
    if (check_varlen(vp, &vs)) return 0;
    return varlen_ws_bytes(vp, vs);
}

int attn_core_fwd_varlen(const attn_core_varlen_params* vp, const void* q, const void* k, const void* v, void* o,
                         float* lse, void* stream)
{
    VarlenShape vs;
    int rc = check_varlen(vp, &vs);
    if (rc) return rc;
    if (!q || !k || !v || !o || !lse) return ATTN_CORE_ERR_INVALID_ARG;
    if (!supported_d(vp->base.d)) return ATTN_CORE_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_CORE_ERR_MISALIGNED;
    if (vs.max_q == 0) return ATTN_CORE_OK;          // no queries: nothing to compute
    const attn_core_params ps = batch_params(vp, vs);
    if ((rc = check_params(&ps))) return rc;
    if ((rc = check_device())) return rc;
    if ((rc = get_encoder())) return rc;
    return fwd_launch(&ps, packed_geometry(vp, vs), q, k, v, o, lse, reinterpret_cast<cudaStream_t>(stream));
}

int attn_core_bwd_varlen(const attn_core_varlen_params* vp, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, void* stream)
{
    VarlenShape vs;
    int rc = check_varlen(vp, &vs);
    if (rc) return rc;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return ATTN_CORE_ERR_INVALID_ARG;
    if (!supported_d(vp->base.d)) return ATTN_CORE_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return ATTN_CORE_ERR_MISALIGNED;
    if (workspace_bytes < varlen_ws_bytes(vp, vs)) return ATTN_CORE_ERR_WORKSPACE_TOO_SMALL;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (vs.max_q == 0) {
        // no query sees any key: every key's gradients are zero
        const size_t nb = (size_t)vs.total_k * vp->base.h_kv * vp->base.d * sizeof(uint16_t);
        if (nb && (cudaMemsetAsync(dk, 0, nb, st) != cudaSuccess || cudaMemsetAsync(dv, 0, nb, st) != cudaSuccess))
            return ATTN_CORE_ERR_CUDA;
        return ATTN_CORE_OK;
    }
    const attn_core_params ps = batch_params(vp, vs);
    if ((rc = check_params(&ps))) return rc;
    if ((rc = check_device())) return rc;
    if ((rc = get_encoder())) return rc;
    return bwd_launch(&ps, packed_geometry(vp, vs), q, k, v, o, lse, dout, dq, dk, dv, workspace, false, st);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Dropout + residual add + layer norm.
namespace {

int check_dal(const attn_core_dal_params* p)
{
    if (p == nullptr) return ATTN_CORE_ERR_INVALID_ARG;
    if (p->n_rows <= 0 || p->hidden <= 0 || p->hidden % 8 != 0) return ATTN_CORE_ERR_INVALID_ARG;
    if (p->hidden > ac::kDalMaxHidden) return ATTN_CORE_ERR_UNSUPPORTED;
    if (!(p->p_drop >= 0.0f && p->p_drop < 1.0f)) return ATTN_CORE_ERR_INVALID_ARG;
    if (!(p->eps > 0.0f) || isinf(p->eps)) return ATTN_CORE_ERR_INVALID_ARG;
    if (p->offset >> 32) return ATTN_CORE_ERR_INVALID_ARG;
    return ATTN_CORE_OK;
}

ac::DalArgs dal_args(const attn_core_dal_params* p)
{
    ac::DalArgs a{};
    a.n_rows = p->n_rows;
    a.hidden = p->hidden;
    a.eps = p->eps;
    a.thr = drop_threshold16(p->p_drop);
    a.keep_scale = 1.0f / (1.0f - (float)a.thr / 65536.0f);
    a.seed_lo = (uint32_t)(p->seed & 0xffffffffu);
    a.seed_hi = (uint32_t)(p->seed >> 32);
    ac::philox_round_keys(a.seed_lo, a.seed_hi, a.rk);
    a.offset = (uint32_t)p->offset;
    a.status = p->dev_status;
    a.timeout_ns = (uint64_t)(p->wait_timeout_ms ? p->wait_timeout_ms : 2000u) * 1000000ull;
    return a;
}

int dal_partial_rows(const attn_core_dal_params* p)
{
    return p->n_rows < ac::kDalMaxPartial ? p->n_rows : ac::kDalMaxPartial;
}

}  // namespace

extern "C" {

int attn_core_dropout_add_ln_fwd(const attn_core_dal_params* p, const void* x, const void* residual,
                                 const float* gamma, const float* beta, void* z, void* y, float* mean,
                                 float* rstd, void* stream)
{
    int rc = check_dal(p);
    if (rc) return rc;
    if (!x || !residual || !gamma || !beta || !z || !y || !mean || !rstd) return ATTN_CORE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(residual) || !aligned16(gamma) || !aligned16(beta) || !aligned16(z) ||
        !aligned16(y))
        return ATTN_CORE_ERR_MISALIGNED;
    if ((rc = check_device())) return rc;
    int sms = 0;
    if ((rc = device_sms(&sms))) return rc;
    ac::DalArgs a = dal_args(p);
    a.x = static_cast<const uint16_t*>(x);
    a.residual = static_cast<const uint16_t*>(residual);
    a.gamma = gamma;
    a.beta = beta;
    a.z = static_cast<uint16_t*>(z);
    a.y = static_cast<uint16_t*>(y);
    a.mean = mean;
    a.rstd = rstd;
    return ac::launch_dal_fwd(a, sms, reinterpret_cast<cudaStream_t>(stream)) ? ATTN_CORE_ERR_CUDA : ATTN_CORE_OK;
}

size_t attn_core_dropout_add_ln_bwd_workspace_bytes(const attn_core_dal_params* p)
{
    if (check_dal(p)) return 0;
    return 2 * sizeof(float) * (size_t)p->hidden * (size_t)dal_partial_rows(p);
}

int attn_core_dropout_add_ln_bwd(const attn_core_dal_params* p, const void* dy, const void* dz_next,
                                 const void* z, const float* mean, const float* rstd, const float* gamma,
                                 void* dx, void* d_residual, float* dgamma, float* dbeta, void* workspace,
                                 size_t workspace_bytes, void* stream)
{
    int rc = check_dal(p);
    if (rc) return rc;
    if (!dy || !z || !mean || !rstd || !gamma || !dx || !d_residual || !dgamma || !dbeta || !workspace)
        return ATTN_CORE_ERR_INVALID_ARG;
    if (!aligned16(dy) || (dz_next && !aligned16(dz_next)) || !aligned16(z) || !aligned16(gamma) ||
        !aligned16(dx) || !aligned16(d_residual) || !aligned16(workspace))
        return ATTN_CORE_ERR_MISALIGNED;
    if (workspace_bytes < attn_core_dropout_add_ln_bwd_workspace_bytes(p)) return ATTN_CORE_ERR_WORKSPACE_TOO_SMALL;
    if ((rc = check_device())) return rc;
    int sms = 0;
    if ((rc = device_sms(&sms))) return rc;
    ac::DalArgs a = dal_args(p);
    a.gamma = gamma;
    a.z = static_cast<uint16_t*>(const_cast<void*>(z));
    a.mean = const_cast<float*>(mean);
    a.rstd = const_cast<float*>(rstd);
    a.dy = static_cast<const uint16_t*>(dy);
    a.dz_next = static_cast<const uint16_t*>(dz_next);
    a.dx = static_cast<uint16_t*>(dx);
    a.d_residual = static_cast<uint16_t*>(d_residual);
    a.dgamma = dgamma;
    a.dbeta = dbeta;
    a.partial = static_cast<float*>(workspace);
    return ac::launch_dal_bwd(a, sms, reinterpret_cast<cudaStream_t>(stream)) ? ATTN_CORE_ERR_CUDA : ATTN_CORE_OK;
}

}  // extern "C"

// GeLU of the layer's MLP.
extern "C" {

int attn_core_gelu_fwd(int64_t n, const void* x, void* y, void* stream)
{
    if (n <= 0 || n % 8 != 0 || !x || !y) return ATTN_CORE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return ATTN_CORE_ERR_MISALIGNED;
    int rc = check_device();
    if (rc) return rc;
    int sms = 0;
    if ((rc = device_sms(&sms))) return rc;
    return ac::launch_gelu_fwd(static_cast<const uint16_t*>(x), static_cast<uint16_t*>(y), n, sms,
                               reinterpret_cast<cudaStream_t>(stream))
               ? ATTN_CORE_ERR_CUDA
               : ATTN_CORE_OK;
}

int attn_core_gelu_bwd(int64_t n, const void* x, const void* dy, void* dx, void* stream)
{
    if (n <= 0 || n % 8 != 0 || !x || !dy || !dx) return ATTN_CORE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(dy) || !aligned16(dx)) return ATTN_CORE_ERR_MISALIGNED;
    int rc = check_device();
    if (rc) return rc;
    int sms = 0;
    if ((rc = device_sms(&sms))) return rc;
    return ac::launch_gelu_bwd(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(dy),
                               static_cast<uint16_t*>(dx), n, sms, reinterpret_cast<cudaStream_t>(stream))
               ? ATTN_CORE_ERR_CUDA
               : ATTN_CORE_OK;
}

}  // extern "C"

// Backward for callers that cannot allocate device memory.  Its workspace is a
// fixed array of this library's own, 2 * kNoAllocMaxRows fp32 values (8 MiB),
// which every GPU that loads the library holds until the process exits.  In
// host code the array's name is only a host-side stand-in: every call looks up
// its device address for the current device with cudaGetSymbolAddress (which
// allocates nothing) and passes that address to the kernels, so the address is
// never stale, not even after the device's context has been reset.
static constexpr size_t kNoAllocMaxRows = (size_t)1 << 20;
static __device__ __align__(256) float g_noalloc_scratch[2 * kNoAllocMaxRows];

extern "C" {

int attn_core_bwd_recompute_noalloc(const attn_core_params* p, const void* q, const void* k, const void* v,
                                    const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                    void* dv, void* stream)
{
    int rc = check_params(p);
    if (rc) return rc;
    if (padded_rows(p) > kNoAllocMaxRows) return ATTN_CORE_ERR_WORKSPACE_TOO_SMALL;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) return ATTN_CORE_ERR_CUDA;
    // The fixed array holds the two row statistics only; the dK/dV kernel draws
    // its own mask.
    return bwd_impl(p, q, k, v, o, lse, dout, dq, dk, dv, addr, sizeof(float) * 2 * kNoAllocMaxRows, false,
                    stream);
}

}  // extern "C"
