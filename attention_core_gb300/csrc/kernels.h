// kernels.h -- internal interface between the C-ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ac {

// Query / key tile height of every kernel (TMEM has 128 lanes).
constexpr int kBlockRows = 128;
// Threads per CTA of the tensor-core kernels: warp 0 loads Q/K (or K/V),
// warp 1 issues MMAs and owns TMEM, warp 2 loads V, warp 3 idles, and warps
// 4..11 are the row threads: two warpgroups that share the 128 TMEM lanes
// (one row per lane) and split every tile's columns in halves, so each SM
// sub-partition runs two of them.
constexpr int kThreads = 384;
constexpr int kRowThreads = 256;
// The dQ kernel adds four warps (12..15) that draw the dropout mask ahead of
// its row threads.
constexpr int kRngThreads = 128;
constexpr int kThreadsRng = kThreads + kRngThreads;
// Register shares after setmaxnreg: row warps / every other warp.  A block
// is launched with (65536 / threads, rounded down to a multiple of 8)
// registers per thread, and the shares must add up to no more than that, or
// the row warps' raise would wait forever; the launcher also checks the
// count the compiler actually gave the kernel.
constexpr int kDqRowRegs = 176, kDqOtherRegs = 80;
constexpr int launch_regs(int threads) { return (65536 / threads) / 8 * 8; }
constexpr int reg_shares(int row_regs, int other_regs, int threads)
{
    return kRowThreads * row_regs + (threads - kRowThreads) * other_regs;
}
static_assert(reg_shares(kDqRowRegs, kDqOtherRegs, kThreadsRng) <= kThreadsRng * launch_regs(kThreadsRng),
              "dQ register shares");

struct CommonArgs {
    int32_t s;            // queries per head
    int32_t s_k;          // keys (and value rows) per KV head; == s when causal
    int32_t h_q, h_kv;    // query / key-value heads
    int32_t n_blk;        // ceil(s / 128): query blocks
    int32_t n_blk_k;      // ceil(s_k / 128): key blocks
    int32_t n_bh;         // b * h_q
    int32_t causal;
    float scale_log2;     // score scale * log2(e)
    float scale;          // score scale
    float keep_scale;     // 1 / (1 - thr / 256)
    uint32_t thr;         // dropout threshold on an 8-bit draw (0: no dropout)
    uint32_t seed_lo, seed_hi, offset;
    uint32_t rk[20];      // Philox key schedule of the seed (philox_round_keys)
    int32_t* status;      // caller-owned device status word (may be null)
    uint64_t timeout_ns;  // limit of every in-kernel wait
    int32_t inject_timeout;  // test hook: every thread waits on a barrier nothing completes
    uint32_t bh0;         // added to the flattened head index in the Philox counter (a
                          // sequence of a packed batch draws as batch element bh0 / h_q)
    int64_t lse_stride;   // LSE elements from one query head to the next (s, or the
                          // packed batch's total query count)
    // Packed (variable-length) batch in one launch: device copies of the
    // sequence tables (n_seq + 1 entries each), or null for the padded layout.
    // Then the batch is n_seq sequences of at most n_blk query blocks and
    // n_blk_k key blocks, n_bh = n_seq * h_q, and every tile takes its own
    // lengths from the tables.
    const int32_t* cu_q;
    const int32_t* cu_k;
    int64_t ws_stride;    // backward workspace rows from one query head to the next:
                          // n_blk * 128 for the padded layout; for a packed batch
                          // the total query count rounded up to 4, plus 132 per
                          // sequence (packed_ws_row0)
};

// First workspace row of sequence `seq` of a packed batch whose queries start
// at row q_first: each sequence's rows padded to whole 128-row blocks, every
// region starting on a multiple of 4 rows (16 bytes, for the bulk copies of
// the dK/dV kernel); the 132-row gap per sequence covers the rounding, so
// regions never overlap.
__host__ __device__ inline int64_t packed_ws_row0(int q_first, int seq)
{
    return (int64_t)((q_first + 3) & ~3) + 132 * (int64_t)seq;
}

// Where one work tile of the query-major kernels (the forward and dQ) lives:
// the query block of one head of one sequence (or batch element), for both
// layouts.  Tile t: query block n_blk - 1 - t / n_bh (longest first), and
// flattened head bh = t % n_bh = sequence * h_q + head.  The kernels are
// compiled for one layout each (PACKED): in the padded one every field follows
// from the launch parameters and `empty` and `tail` are constant false, so the
// packed batch's bookkeeping costs the padded kernels nothing.
struct QTile {
    int qb;          // query block within its sequence
    int bh;          // flattened query head (Philox counter word 2, minus bh0)
    int bkv;         // flattened KV head
    int nk;          // key blocks of width BN to visit
    int yq, zq;      // TMA row / head coordinates of the tile's first query row
    int yk, zk;      // TMA row / head coordinates of the sequence's first key row
    int lq, lk;      // queries and keys of the sequence
    int64_t ws0;     // workspace row of the tile's first query row
    bool empty;      // a packed batch's tile past its sequence's end: no work
    bool tail;       // a packed batch's tile that holds rows past its sequence's
                     // end (they are not stored: the next sequence follows)
};
template <bool PACKED>
__device__ __forceinline__ QTile q_tile(const CommonArgs& a, int t, int bn)
{
    QTile w;
    w.qb = a.n_blk - 1 - t / a.n_bh;
    w.bh = t % a.n_bh;
    const int group = a.h_q / a.h_kv;
    const int seq = w.bh / a.h_q, head = w.bh % a.h_q;
    w.bkv = seq * a.h_kv + head / group;
    if constexpr (!PACKED) {
        w.lq = a.s;
        w.lk = a.s_k;
        w.yq = w.qb * 128;
        w.zq = w.bh;
        w.yk = 0;
        w.zk = w.bkv;
        w.ws0 = (int64_t)w.bh * a.ws_stride + w.qb * 128;
        w.empty = false;
        w.tail = false;
    } else {
        const int q0 = a.cu_q[seq], k0 = a.cu_k[seq];
        w.lq = a.cu_q[seq + 1] - q0;
        w.lk = a.cu_k[seq + 1] - k0;
        w.yq = q0 + w.qb * 128;
        w.zq = head;
        w.yk = k0;
        w.zk = head / group;
        w.ws0 = (int64_t)head * a.ws_stride + packed_ws_row0(q0, seq) + w.qb * 128;
        w.empty = w.qb * 128 >= w.lq;
        w.tail = (w.qb + 1) * 128 > w.lq;
    }
    const int n_kblk = (w.lk + bn - 1) / bn;
    const int nk_causal = (w.qb + 1) * (128 / bn);
    w.nk = w.empty ? 0 : (a.causal ? (nk_causal < n_kblk ? nk_causal : n_kblk) : n_kblk);
    return w;
}

struct FwdArgs {
    CommonArgs c;
    uint16_t* o;          // bf16 [b*h_q*s*d], or a packed [tokens, h_q, d]
    float* lse;           // tile row r at lse[zq * c.lse_stride + yq + r] (QTile)
    int64_t o_head_stride, o_row_stride;   // elements, for O stored row by row (d = 160,
                                           // and a packed batch's tail tiles): tile row r
                                           // at o + zq * head + (yq + r) * row
    int32_t num_sms;      // persistent grid size
};

struct BwdArgs {
    CommonArgs c;
    int32_t s_pad;        // n_blk * 128
    const uint16_t* o;    // bf16 [b*h_q*s*d]
    const uint16_t* dout; // bf16 [b*h_q*s*d]
    const float* lse;     // [b*h_q*s]
    float* lse2_ws;       // [b*h_q*s_pad]  -LSE * log2(e); -inf past s
    float* delta_ws;      // [b*h_q*s_pad]  minus the exact row statistic D = sum_j P_ij dP_ij
                          // (written by the dQ kernel, read by the dK/dV kernel)
    uint32_t* mask_ws;    // dropout keep bits, written by the dQ kernel and read by the
                          // dK/dV kernel (layout: mask_pair_word); null: dK/dV draws its own
    int32_t d;
    int32_t num_sms;      // persistent grid size
    // For rows stored one by one (a packed batch's tail tiles): the gradients
    // and their strides in elements, as FwdArgs::o.
    uint16_t* dq;
    uint16_t* dk;
    uint16_t* dv;
    int64_t q_head_stride, q_row_stride, kv_head_stride, kv_row_stride;
};

// Keep bits handed from the dQ kernel to the dK/dV kernel.  For every
// (query head, 128-query block qb, 128-key block kb) that the causal mask does
// not hide, two 1 KB units (query rows 0-63 and 64-127 of the block); unit
// word [g * 64 + row] holds whether the pairs (query row, key 32 g + c of the
// block) are kept, key c at bit keep_bit_position(c) (philox.cuh).  Returns
// the index of the pair's first word.
__host__ __device__ inline size_t mask_pair_word(const CommonArgs& a, int bh, int qb, int kb)
{
    const size_t per_head = a.causal ? (size_t)a.n_blk * (a.n_blk + 1) / 2 : (size_t)a.n_blk * a.n_blk_k;
    const size_t pair = a.causal ? (size_t)qb * (qb + 1) / 2 + kb : (size_t)qb * a.n_blk_k + kb;
    return ((size_t)bh * per_head + pair) * 512;
}
inline size_t mask_ws_words(const CommonArgs& a) { return mask_pair_word(a, a.n_bh, 0, 0); }

// Host launchers; return a cudaError_t value.
int launch_fwd(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream);
int launch_bwd_dkdv(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk,
                    const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                    const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t stream);
int launch_bwd_dq(int d, bool dropout, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const CUtensorMap& tdo, const CUtensorMap& to, const CUtensorMap& tdq, const BwdArgs& a,
                  cudaStream_t stream);

// Dropout + residual add + layer norm (dropout_add_ln.cu).  Rows are tokens,
// `hidden` (a multiple of 8) the row length; bf16 tensors are row-major.
struct DalArgs {
    int32_t n_rows, hidden;
    float eps;
    float keep_scale;     // 1 / (1 - thr / 65536)
    uint32_t thr;         // dropout threshold on a 16-bit draw (0: no dropout)
    uint32_t seed_lo, seed_hi, offset;
    uint32_t rk[20];             // Philox key schedule of the seed (philox_round_keys)
    const uint16_t* x;           // fwd: sub-layer output entering the dropout
    const uint16_t* residual;    // fwd
    const float* gamma;          // fwd, bwd
    const float* beta;           // fwd
    uint16_t* z;                 // fwd: written; bwd: read
    uint16_t* y;                 // fwd
    float* mean;                 // fwd: written; bwd: read
    float* rstd;                 // fwd: written; bwd: read
    const uint16_t* dy;          // bwd
    const uint16_t* dz_next;     // bwd, may be null
    uint16_t* dx;                // bwd
    uint16_t* d_residual;        // bwd
    float* dgamma;               // bwd
    float* dbeta;                // bwd
    float* partial;              // bwd workspace: [2][grid][hidden] per-CTA column sums
    int32_t* status;             // caller-owned device status word (may be null)
    uint64_t timeout_ns;         // limit of every in-kernel wait
};
constexpr int kDalMaxHidden = 28672;   // backward keeps 8 * hidden bytes of column sums in shared memory
constexpr int kDalMaxPartial = 320;   // backward CTAs (rows of the partial-sum workspace)
// Grids are sized from the device's SM count and each kernel's occupancy.
int launch_dal_fwd(const DalArgs& a, int sms, cudaStream_t stream);
int launch_dal_bwd(const DalArgs& a, int sms, cudaStream_t stream);

// GeLU (tanh form) of the layer's MLP, elementwise on n bf16 values (n % 8 == 0).
int launch_gelu_fwd(const uint16_t* x, uint16_t* y, int64_t n, int sms, cudaStream_t stream);
int launch_gelu_bwd(const uint16_t* x, const uint16_t* dy, uint16_t* dx, int64_t n, int sms, cudaStream_t stream);

// Query-tile height of the dK/dV kernel for head dimension d (TMEM budget).
constexpr int dkdv_query_tile(int d) { return (2 * d + 2 * 128 <= 512) ? 128 : 64; }
// Key-block width of the dQ kernel for head dimension d (TMEM budget:
// S, dP, and two d-wide accumulators).
constexpr int dq_key_tile(int d) { return (2 * 128 + 2 * d <= 512) ? 128 : 64; }

}  // namespace ac
