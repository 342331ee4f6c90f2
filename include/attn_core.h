/*
 * attn_core.h -- C ABI of the GB300 (sm_103a) attention-core library.
 *
 * The attention core is QK^T, softmax, softmax dropout and attention over V:
 * the part of a transformer layer that selective activation recomputation
 * does not store, because its activations are large and its FLOPs few, and
 * recomputes in the backward pass instead ("Reducing Activation
 * Recomputation in Large Transformer Models", dmarx anthology LIT-736, Key
 * takeaways, fourth bullet; "Recomputing Activations", curionode Plate 2,
 * second paragraph and "Memory for compute, selectively").
 *
 * attn_core_fwd stores only O and one fp32 log-sum-exp per query row; with
 * Q, K, V and the Philox seed/offset that is everything the backward pass
 * needs.  attn_core_bwd_recompute rebuilds the scores, probabilities and
 * dropout mask on chip and never writes them to global memory, so the
 * 5 a s^2 b byte term of the per-layer activation formula sbh(34 + 5as/h)
 * is never held in device memory.  attn_core_stored_bytes reports that
 * accounting exactly.
 *
 * Tensors (all device pointers, 16-byte aligned, contiguous, row-major):
 *   Q, O, dO, dQ : bf16 [b, h_q,  s,    d]
 *   K, V, dK, dV : bf16 [b, h_kv, s_kv, d]   (s_kv = s unless set)
 *   LSE          : fp32 [b, h_q, s]   natural-log log-sum-exp of each row
 * Query head h uses KV head h / (h_q / h_kv) (grouped-query attention).
 * Causal masking is top-left aligned: query i sees keys 0..i; it needs
 * s_kv == s.  Without it, s queries attend to all s_kv keys
 * (cross-attention when s_kv != s).
 *
 * Readings the pages leave open (the CPU oracle in the tests follows the
 * same ones):
 *   - scale: scale <= 0 selects 1/sqrtf(d), computed in fp32.
 *   - LSE is in natural-log units.
 *   - dropout acts on the normalised probabilities, before the product with V.
 *   - dropout mask: Philox-4x32-10 (Salmon et al., SC'11) with key
 *     (seed & 0xffffffff, seed >> 32) and counter (j / 16, i, b*h_q + h,
 *     offset) for query i, key j of query head h in batch b; the call's four
 *     output words give sixteen 8-bit draws, key j taking byte j % 4 (bits
 *     8 (j % 4) .. 8 (j % 4) + 7) of word (j % 16) / 4.  With
 *     thr = round(p * 256) (at most 255) an element is dropped iff its draw <
 *     thr, and kept elements are scaled by 1 / (1 - thr / 256): the effective
 *     rate is p rounded to a multiple of 1/256 (p = 0.1 drops 26/256 =
 *     0.1015625 of the elements; p < 1/512 drops none).  p == 0 draws nothing.
 *
 * Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  The library allocates no device memory: the caller owns
 * every buffer, including the backward workspace.
 */
#ifndef ATTN_CORE_H
#define ATTN_CORE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  On any non-zero code no kernel has been launched and no
 * output has been written, except ATTN_CORE_ERR_CUDA from a launch, which
 * reports the CUDA error of that launch. */
#define ATTN_CORE_OK 0
#define ATTN_CORE_ERR_INVALID_ARG 1         /* null pointer, bad shape, p outside [0,1), offset >= 2^32 */
#define ATTN_CORE_ERR_UNSUPPORTED 2         /* head dimension or device not supported */
#define ATTN_CORE_ERR_MISALIGNED 3          /* a pointer is not 16-byte aligned (workspace: 256) */
#define ATTN_CORE_ERR_WORKSPACE_TOO_SMALL 4 /* bwd workspace smaller than attn_core_bwd_workspace_bytes */
#define ATTN_CORE_ERR_CUDA 5                /* a CUDA runtime or driver call failed */
#define ATTN_CORE_ERR_DEVICE_TIMEOUT 6      /* a kernel wait ran past its limit (reported via dev_status) */

/* flags */
#define ATTN_CORE_FLAG_REDRAW_MASK 0x1         /* backward: the dK/dV kernel draws the dropout mask again
                                                  instead of reading keep bits the dQ kernel wrote to the
                                                  workspace; the workspace then holds only the row
                                                  statistics (smaller, see attn_core_bwd_workspace_bytes)
                                                  at the cost of a second Philox pass */
#define ATTN_CORE_FLAG_TEST_WAIT_TIMEOUT 0x100 /* test hook: every kernel waits on a barrier that nothing
                                                  completes; it gives up after wait_timeout_ms, writes
                                                  ATTN_CORE_ERR_DEVICE_TIMEOUT to dev_status and exits */

typedef struct {
    int32_t b, h_q, h_kv, s, d; /* s queries per head; h_q % h_kv == 0; d in {64, 96, 128, 160} */
    int32_t causal;             /* 0 or 1 */
    float p_drop;               /* softmax-dropout probability in [0, 1) */
    float scale;                /* score scale; <= 0 selects 1/sqrtf(d) */
    uint64_t seed;              /* Philox key */
    uint64_t offset;            /* Philox counter word 3; must be < 2^32 */
    /* Optional caller-owned device int32, zero before the call.  A kernel
     * whose wait runs out writes (ATTN_CORE_ERR_DEVICE_TIMEOUT | site << 8)
     * there (first error wins); read it after synchronising.  May be NULL. */
    int32_t* dev_status;
    int32_t flags;              /* ATTN_CORE_FLAG_* */
    uint32_t wait_timeout_ms;   /* limit of each in-kernel wait; 0 selects 2000 ms */
    /* Optional profiling hook: an array of cudaEvent_t handles, two per
     * kernel the call launches (fwd: 1 kernel; bwd: 2 kernels, in order
     * dQ, dK/dV), recorded on `stream` immediately before and
     * after each launch.  May be NULL. */
    void** timing_events;
    /* Keys (and value rows) per KV head; 0 selects s.  With s_kv != s the
     * causal mask is aligned top-left: query i sees keys 0 .. min(i, s_kv - 1)
     * (with more keys than queries, keys s .. s_kv - 1 are seen by no query
     * and get zero dK and dV).  The dropout mask of (query i, key j) does not
     * depend on s or s_kv. */
    int32_t s_kv;
} attn_core_params;

typedef struct {
    /* Per-layer activation bytes of one rank's shard, hidden h = h_q * d:
     * the activation-checkpointing page's per-token forms 34d + 5HT,
     * 34d and 2d ("Recomputing Activations", Workshop) times s * b. */
    int64_t layer_none;           /* 34 s b h + 5 h_q s^2 b : nothing recomputed */
    int64_t layer_selective;      /* 34 s b h               : attention core recomputed */
    int64_t layer_full;           /* 2 s b h                : only the layer input kept */
    int64_t core_scores_avoided;  /* 5 h_q s s_kv b         : what this library never stores */
    int64_t core_kept;            /* 2 d b (2 h_q s + 2 h_kv s_kv): Q, K, V, O in bf16 */
    int64_t core_recompute_state; /* 4 b h_q s + 16         : LSE and seed/offset */
} attn_core_bytes;

/* Forward: O and LSE from Q, K, V (the core's forward in the takeaways'
 * order: QK^T, softmax, softmax dropout, attention over V).  Launches one
 * kernel.  Writes O and LSE only. */
int attn_core_fwd(const attn_core_params* p, const void* q, const void* k, const void* v, void* o,
                  float* lse, void* stream);

/* Bytes of device workspace attn_core_bwd_recompute needs, 0 if p is invalid:
 *   8 * b * h_q * ceil(s / 128) * 128   two fp32 row statistics per padded
 *                                       query row, and, when p_drop > 0 and
 *                                       d <= 128,
 *   2048 * b * h_q * N                  the dropout keep bits, one bit per
 *                                       (query, key) of each 128 x 128 block,
 * with N = n (n + 1) / 2 blocks per head if causal with s_kv == s
 * (n = ceil(s / 128)), ceil(s / 128) * ceil(s_kv / 128) if not causal, and no
 * keep bits for causal with s_kv != s (the second kernel draws the mask again).  The keep bits are transient (written and
 * read within one backward call) but scale with s^2: 6.7 MB for b = 2,
 * h_q = 12, s = 2048, and 272 MB for h_q = 64, s = 8192.  Callers short of
 * memory set ATTN_CORE_FLAG_REDRAW_MASK to leave them out. */
size_t attn_core_bwd_workspace_bytes(const attn_core_params* p);

/* Backward with recomputation: dQ, dK, dV from Q, K, V, O, LSE and dO.  The
 * scores, probabilities and dropout mask are rebuilt on chip from Q, K, LSE
 * and (seed, offset); the mask is bit-identical to the forward's.  For
 * d <= 128 it is drawn once, by the first kernel, which hands it to the
 * second as bits in the workspace (nothing of it outlives the call); for
 * d = 160 each kernel draws it.  The
 * softmax row statistic sum_j P_ij dP_ij is formed exactly from the
 * recomputed P and dP (a first estimate from the stored bf16 O is corrected
 * in fp32), not rounded through the stored output.  Launches two kernels
 * (dQ with the row statistics, then dK/dV).  `workspace` is caller-owned
 * device memory of at least attn_core_bwd_workspace_bytes(p) bytes, 256-byte
 * aligned; its contents on entry do not matter.  dQ, dK, dV are written
 * whole (no accumulation into existing contents). */
int attn_core_bwd_recompute(const attn_core_params* p, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Backward with recomputation for callers that cannot allocate device
 * memory.  Some callers have no allocator to call: code running inside
 * another framework that owns every byte of device memory through its own
 * pool, code invoked from a library that forbids allocation in its callbacks,
 * or services whose memory is planned once at start-up.  They cannot provide
 * the workspace attn_core_bwd_recompute asks for, so this variant uses a
 * fixed scratch array inside the library instead and allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine).  The paper
 * has no counterpart to this entry point.
 *
 * Same arguments and results as attn_core_bwd_recompute without the
 * workspace.  The array holds the row statistics only, so here the second
 * kernel draws the dropout mask again from Philox (the same bits).  Limit: b * h_q * ceil(s / 128) * 128 <= 1048576 padded query
 * rows (the array holds 8 MiB on every GPU that loads the library, until the
 * process exits); larger shapes return ATTN_CORE_ERR_WORKSPACE_TOO_SMALL
 * without launching anything.  Every call looks up the array's device
 * address for the current device (cudaGetSymbolAddress, which allocates
 * nothing); the first call on a device may make the runtime load this
 * library's device code there, so make that first call before any stream
 * capture.  All calls on a device
 * share the one array and it keeps the last call's contents (nothing in it
 * needs to start at zero), so calls whose kernels overlap on the GPU --
 * concurrent streams, or several host threads -- race on it: order them. */
int attn_core_bwd_recompute_noalloc(const attn_core_params* p, const void* q, const void* k, const void* v,
                                    const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                    void* dv, void* stream);

/* ------------------------------------------------------------------------
 * Variable-length (packed) batches.  n_seq sequences of different lengths in
 * one token-major tensor; the tokens of sequence i are rows cu_seqlens_q[i]
 * .. cu_seqlens_q[i + 1] - 1 (keys: cu_seqlens_k, NULL for the same table):
 *   Q, O, dO, dQ : bf16 [total_q, h_q, d]     total_q = cu_seqlens_q[n_seq]
 *   K, V, dK, dV : bf16 [total_k, h_kv, d]
 *   LSE          : fp32 [h_q, total_q]
 * Each sequence attends only within itself, as batch element i of the
 * padded layout would: the same causal rule (top-left aligned when a
 * sequence's query and key counts differ), and the same dropout mask
 * (Philox counter word 2 = i * h_q + head).  The sequence tables are arrays
 * of n_seq + 1 int32 starting at 0 and nondecreasing, given twice: in host
 * memory (cu_seqlens_q / _k: checked, and used to size the launch) and as a
 * device copy with the same values (cu_seqlens_q_dev / _k_dev, read by the
 * kernels; _k_dev may be NULL only when cu_seqlens_k is).  An empty sequence
 * is skipped, one with queries but no keys is invalid; one with keys but no
 * queries gets zero dK and dV rows.  `base` supplies h_q, h_kv, d, causal,
 * p_drop, scale, seed, offset, dev_status, flags and wait_timeout_ms; its b,
 * s and s_kv are ignored and its timing_events must be NULL.  The whole
 * batch is one launch per kernel (the same kernels as the padded entry
 * points): they take the batch as n_seq elements of the longest sequence's
 * length, skip the work past each sequence's end, and store the rows of a
 * sequence's last, partial block one by one so that nothing lands in the next
 * sequence.  Both tables must stay unchanged until the calls' kernels have
 * run. */
typedef struct {
    attn_core_params base;
    int32_t n_seq;
    const int32_t* cu_seqlens_q;       /* host, n_seq + 1 */
    const int32_t* cu_seqlens_k;       /* host, n_seq + 1, or NULL: as cu_seqlens_q */
    const int32_t* cu_seqlens_q_dev;   /* device copy of cu_seqlens_q */
    const int32_t* cu_seqlens_k_dev;   /* device copy of cu_seqlens_k, or NULL with it */
} attn_core_varlen_params;

int attn_core_fwd_varlen(const attn_core_varlen_params* p, const void* q, const void* k, const void* v, void* o,
                         float* lse, void* stream);

/* Workspace of attn_core_bwd_varlen, 0 if p is invalid: the two fp32 row
 * statistics of every query row, each sequence's rows padded to whole
 * 128-row blocks and aligned to 16 bytes:
 * 8 * h_q * (round_up(total_q, 4) + 132 * n_seq) bytes, rounded up to 256.
 * (The dropout mask is drawn twice in a packed batch; there are no keep bits.) */
size_t attn_core_bwd_varlen_workspace_bytes(const attn_core_varlen_params* p);

int attn_core_bwd_varlen(const attn_core_varlen_params* p, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Activation-byte accounting (pure host, integer, exact).  Worked example of
 * the activation-checkpointing page: Llama 3 70B, s = 8192, b = 1, h_q = 64,
 * d = 128, 80 layers -> 1.9 TB none, 182.5 GB selective, 10.7 GB full. */
int attn_core_stored_bytes(const attn_core_params* p, attn_core_bytes* out);

/* Static description of a return code. */
const char* attn_core_strerror(int code);

/* ------------------------------------------------------------------------
 * Dropout + residual add + layer norm at a residual sub-layer boundary, on
 * either side of the attention core.  These are the layer norms and the
 * dropouts after the attention block and the MLP that tensor parallelism
 * leaves replicated and that act on each sequence position independently
 * ("Reducing Activation Recomputation in Large Transformer Models", dmarx
 * anthology LIT-736, Key takeaways, first and second bullets).  Reading of
 * the block (the pages give no formula), per row (token) of `hidden` values:
 *     z = residual + dropout(x)                            stored, bf16
 *     y = gamma * (z - mean) * rstd + beta                 bf16
 *     rstd = 1 / sqrt(var + eps), var the biased variance of the stored z.
 * Dropout mask: Philox-4x32-10 with the core's key, counter (col / 8, row,
 * 0xFFFFFFFF, offset) (word 2 is a value no attention head index takes) and
 * eight 16-bit draws per call, column col taking the low (col even) or high
 * (col odd) half of word (col % 8) / 2; dropped iff the draw <
 * round(p * 65536) (at most 65535), kept values scaled by
 * 1 / (1 - thr / 65536).  This block is bound by memory traffic, not by the
 * generator, so it keeps the finer 16-bit draws.  As
 * in the core, the backward redraws the mask from (seed, offset); the block
 * keeps z, mean and rstd only.
 *
 * Tensors (device pointers, 16-byte aligned, contiguous, row-major):
 *   x, residual, z, y, dy, dz_next, dx, d_residual : bf16 [n_rows, hidden]
 *   gamma, beta, dgamma, dbeta                      : fp32 [hidden]
 *   mean, rstd                                      : fp32 [n_rows]
 * Asynchronous on `stream`; nothing is allocated.  Return codes as above. */
typedef struct {
    int32_t n_rows;   /* tokens, >= 1 */
    int32_t hidden;   /* multiple of 8, 8 .. 28672 */
    float p_drop;     /* [0, 1) */
    float eps;        /* layer-norm epsilon, > 0 */
    uint64_t seed;    /* Philox key */
    uint64_t offset;  /* Philox counter word 3; must be < 2^32 */
    /* Optional caller-owned device int32, zero before the call: a forward
     * wait that runs out writes ATTN_CORE_ERR_DEVICE_TIMEOUT | 1 << 8 there.
     * May be NULL. */
    int32_t* dev_status;
    uint32_t wait_timeout_ms;   /* limit of each in-kernel wait; 0 selects 2000 ms */
} attn_core_dal_params;

/* Forward: writes z, y, mean and rstd.  Launches one kernel. */
int attn_core_dropout_add_ln_fwd(const attn_core_dal_params* p, const void* x, const void* residual,
                                 const float* gamma, const float* beta, void* z, void* y, float* mean,
                                 float* rstd, void* stream);

/* Bytes of device workspace the backward needs: 8 * hidden * min(n_rows, 320)
 * (per-CTA column sums for dgamma and dbeta), 0 if p is invalid. */
size_t attn_core_dropout_add_ln_bwd_workspace_bytes(const attn_core_dal_params* p);

/* Backward from dy (gradient of y) and, optionally, dz_next (the gradient
 * reaching z through the residual path; NULL for none):
 *     dz = rstd * (g - mean(g) - xhat * mean(g * xhat)) + dz_next,
 *          g = dy * gamma, xhat = (z - mean) * rstd,
 *     d_residual = dz,  dx = dz * keep / (1 - p_eff),
 *     dgamma = sum over rows of dy * xhat,  dbeta = sum over rows of dy.
 * Needs z, mean and rstd from the forward, not x or residual.  dgamma and
 * dbeta are summed in a fixed order (bit-reproducible).  Launches two
 * kernels; `workspace` is caller-owned device memory of at least
 * attn_core_dropout_add_ln_bwd_workspace_bytes(p) bytes, 16-byte aligned. */
int attn_core_dropout_add_ln_bwd(const attn_core_dal_params* p, const void* dy, const void* dz_next,
                                 const void* z, const float* mean, const float* rstd, const float* gamma,
                                 void* dx, void* d_residual, float* dgamma, float* dbeta, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * GeLU of the layer's MLP, for the layer-level measurement of selective
 * recomputation (the anthology page's Key takeaways, fourth bullet: recompute
 * the whole layer, or only the attention core).  Tanh form:
 *     y = x / 2 * (1 + tanh(sqrt(2 / pi) * (x + 0.044715 x^3))),
 * elementwise on n bf16 values (n a multiple of 8, pointers 16-byte aligned),
 * fp32 arithmetic.  The backward writes dx = dy * dy/dx at x.  One kernel
 * each, asynchronous on `stream`. */
int attn_core_gelu_fwd(int64_t n, const void* x, void* y, void* stream);
int attn_core_gelu_bwd(int64_t n, const void* x, const void* dy, void* dx, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_CORE_H */
