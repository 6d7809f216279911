/*
 * attn.h — C ABI of libattn_gb300.so: exact fused scaled-dot-product
 * attention in bf16 for NVIDIA GB300 (sm_103a), forward and backward.
 *
 * What is computed (all entry points): for every (batch or sequence, head),
 *   a_ij  = softmax_scale * q_i . k_j        for visible keys j, -inf otherwise
 *   O_i   = sum_j softmax_j(a_i) v_j,        LSE_i = log sum_j exp(a_ij)
 * and, in the backward entry points, the gradients of <O, dO>:
 *   P = exp(a - LSE), dV = P^T dO, dP = dO V^T, D_i = dO_i . O_i,
 *   dS = P * (dP - D), dQ = scale * dS K, dK = scale * dS^T Q.
 * This is exact attention; the tiled online softmax that computes it is the
 * one of the FlashAttention series (ainexis deep-dive "Tri Dao
 * FlashAttention-4", section 背景), with the conditional rescaling of wittx
 * "FlashAttention-4", section 90%的rescaling都是白干的 (rescale only when a
 * row's max grows by more than 8.0 in log2 units, exact final normalisation),
 * and exp2 split between the hardware unit and a Cody-Waite + cubic polynomial
 * on the FMA pipe (same page, section 用软件"伪造"硬件指令).
 *
 * Visibility. Key j (of a sequence of Nk keys) is visible to query i (of Nq
 * queries) iff j < Nk and, when causal != 0, j <= i + (Nk - Nq) (causal mask
 * aligned to the bottom-right corner; equals j <= i when Nq == Nk). A query
 * row that sees no key gets O = 0, LSE = -inf and zero gradient.
 *
 * Layouts (all element counts, not bytes). Dense tensors are 4-D
 * [batch, seqlen, heads, head_dim] addressed as
 *   base + b*batch_stride + n*row_stride + h*head_stride + d,
 * i.e. head_dim must be contiguous. Variable-length ("varlen") tensors are
 * packed [total_tokens, heads, head_dim]: the batch stride is ignored and
 * sequence s occupies rows cu_seqlens[s] .. cu_seqlens[s+1]-1.
 * LSE is fp32, natural log, contiguous [batch, heads, seqlen_q] (dense) or
 * [heads, total_q] (varlen).
 *
 * Requirements (else ATTN_ERR_INVALID_ARG, nothing launched):
 *   - (d_qk, d_v) in {(64,64), (128,128), (192,128)}  (else ATTN_ERR_UNSUPPORTED);
 *   - q, k, v, o, dO, dQ, dK, dV base addresses 16-byte aligned, every stride a
 *     multiple of 8 elements (16 bytes), lse 4-byte aligned;
 *   - softmax_scale finite and > 0; batch, heads >= 1; seqlens >= 0.
 *
 * Ownership and execution. Every pointer in the parameter structs is a
 * DEVICE pointer owned by the caller; the library never allocates, frees or
 * keeps a pointer after the call returns. Scratch memory ("workspace") is
 * passed in by the caller: query its size with the *_workspace_size call;
 * a workspace may be reused by calls that are ordered on the same stream but
 * must not be shared by calls that can run concurrently. Calls are
 * asynchronous on `stream`: a return of ATTN_OK means the work was enqueued.
 * Kernel-side failures (a bounded wait that gave up) are recorded in a
 * per-process device status word, read (and cleared) by
 * attn_get_device_status. All entry points are thread-safe for distinct
 * output buffers.
 *
 * Devices. Each call runs on the device that owns its tensors: it makes that
 * device current on the calling thread for the duration of the call and then
 * restores the thread's previous current device (when that device's context
 * already exists; the call never creates a context on another GPU).
 */
#ifndef ATTN_GB300_H_
#define ATTN_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 5

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride, alignment or scale */
  ATTN_ERR_UNSUPPORTED = 2,  /* head-dim combination not built */
  ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (see attn_last_cuda_error) */
  ATTN_ERR_TIMEOUT = 4,      /* a kernel's bounded wait gave up (device status word) */
  ATTN_ERR_WORKSPACE = 5     /* workspace missing or smaller than *_workspace_size */
} attn_status_t;

/* Score modifications (attn_fwd_params.score_mod). */
typedef enum {
  ATTN_SCORE_NONE = 0,
  ATTN_SCORE_SOFTCAP = 1,  /* a' = softcap * tanh(a / softcap) */
  ATTN_SCORE_ALIBI = 2     /* a' = a - m_h * |j - (i + Nk - Nq)| */
} attn_score_mod_t;

/* Element type of q, k, v (attn_fwd_params.input_dtype). */
typedef enum {
  ATTN_INPUT_BF16 = 0,
  ATTN_INPUT_E4M3 = 1  /* FP8 E4M3 codes (1 byte each), with per-tensor descale factors */
} attn_input_dtype_t;

/* Opaque CUDA stream handle (cudaStream_t); NULL is the legacy default stream. */
typedef void* attn_stream_t;

/* Forward parameters. Inputs q, k, v (bf16); outputs o (bf16) and lse (fp32).
 * Dense: batch, seqlen_q, seqlen_k describe [batch, seqlen, heads, d] tensors
 * and cu_seqlens_q / cu_seqlens_k must be NULL. Varlen: cu_seqlens_q and
 * cu_seqlens_k are device int32 arrays of num_seqs+1 non-decreasing offsets
 * starting at 0; total_q / total_k are the packed row counts (= last offset),
 * max_seqlen_q / max_seqlen_k bound every sequence's length; batch and the
 * batch strides are ignored. Work scheduling (the tile scheduler for
 * variable-length balance of newton wiki "FlashAttention-4", 核心技術): when
 * max_seqlen_q <= 2047 x 256 (forward), or max_seqlen_q and max_seqlen_k <=
 * 2047 x 128 (backward, per kernel), the call first builds on the stream, in
 * its workspace, a list with one entry per real block of rows, the sequences
 * with the most blocks first, and launches one CTA per entry; otherwise each
 * sequence gets a grid slice sized for max_seqlen. The results are the same
 * bits either way. */
typedef struct attn_fwd_params {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t q_batch_stride, q_row_stride, q_head_stride;
  int64_t k_batch_stride, k_row_stride, k_head_stride;
  int64_t v_batch_stride, v_row_stride, v_head_stride;
  int64_t o_batch_stride, o_row_stride, o_head_stride;
  int32_t batch;
  int32_t heads;
  int32_t seqlen_q;
  int32_t seqlen_k;
  int32_t d_qk;
  int32_t d_v;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int32_t num_seqs;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  int32_t total_q;
  int32_t total_k;
  float softmax_scale;
  int32_t causal;
  /* Forward only: share of exp2 computed on the FMA pipe by the Cody-Waite
   * split + cubic instead of the hardware unit: 0 (none), 8 (one column in
   * eight of every row) or 4 (one in four); anything else is
   * ATTN_ERR_INVALID_ARG. The pages balance the two units for a part with
   * half of GB300's ex2 throughput; on GB300 0 is fastest. Ignored by the
   * backward entry points. */
  int32_t exp2_emu_period;
  /* Optional (may be NULL): device uint64[2] to which the forward kernel adds
   * the number of conditional rescales performed after a row's first key
   * tile ([0]) and the number of such rescale opportunities ([1]). */
  unsigned long long* rescale_stats;
  /* Score modification (the FlexAttention variants built on FA4: wittx
   * "FlashAttention-4", section Python写GPU内核), applied to the scaled logit
   * a = softmax_scale * q_i . k_j of every visible (query i, key j) before the
   * softmax, i and j counted within the sequence; LSE is that of the modified
   * logits and the backward differentiates through the modification:
   *   ATTN_SCORE_NONE: a unchanged (softcap and alibi_slopes are ignored);
   *   ATTN_SCORE_SOFTCAP: a' = softcap * tanh(a / softcap), softcap finite and
   *     > 0 (else ATTN_ERR_INVALID_ARG); the backward multiplies dS by
   *     1 - tanh^2(a / softcap);
   *   ATTN_SCORE_ALIBI: a' = a - m_h |j - (i + Nk - Nq)|, m_h = alibi_slopes[h],
   *     a device float[heads] on q's GPU, 4-byte aligned (else
   *     ATTN_ERR_INVALID_ARG), each finite and >= 0 (the kernels use |m_h|).
   * A modification needs exp2_emu_period == 0 and, in the backward,
   * cta_pair == 0 (else ATTN_ERR_UNSUPPORTED); any other value of score_mod
   * is ATTN_ERR_INVALID_ARG. */
  int32_t score_mod;
  float softcap;
  const float* alibi_slopes;
  /* Element type of q, k and v (the FP8 path of FA3 and the lower precisions
   * named for later versions: ainexis "Tri Dao FlashAttention-4", 背景; wittx
   * "FlashAttention-4", closing section). ATTN_INPUT_BF16 (0, the descales are
   * ignored) or ATTN_INPUT_E4M3 (1): q, k, v hold FP8 E4M3 codes (OCP FP8,
   * 1 byte per element, bias 7, max 448) standing for code * q_descale,
   * code * k_descale and code * v_descale; each descale finite and > 0 (else
   * ATTN_ERR_INVALID_ARG). E4M3 is a forward-only type (attn_fwd and
   * attn_fwd_varlen) for d_qk = d_v = 128, exp2_emu_period 0 and no score
   * modification; other uses, the block-sparse forward and every backward
   * entry point give ATTN_ERR_UNSUPPORTED. Strides (in elements = bytes) must
   * be multiples of 16. O (bf16) and LSE (fp32) are as for bf16 inputs: the
   * result of attention on the dequantised values. Other values of
   * input_dtype are ATTN_ERR_INVALID_ARG. */
  int32_t input_dtype;
  float q_descale;
  float k_descale;
  float v_descale;
  /* Forward only (the backward's own cta_pair field selects its kernel):
   * cta_pair != 0 runs the forward over clusters of two CTAs, the two-SM MMA
   * (M = 256 pair) of wittx "FlashAttention-4", sections 反向传播的优化 and
   * Blackwell的跛脚问题: each CTA holds 128 rows of a 256-row query tile and
   * loads half of every K and V tile. Same results within rounding. Only
   * d_qk = d_v = 128, bf16 inputs, exp2_emu_period 0, no score modification,
   * dense or varlen, not block-sparse (else ATTN_ERR_UNSUPPORTED); varlen
   * then launches from the block index (no tile list). The default (0) is
   * the one-SM kernel, the faster of the two on GB300. */
  int32_t cta_pair;
} attn_fwd_params;

/* Backward parameters. `fwd` holds q, k, v, the forward's outputs o and lse
 * (read-only here), shapes, scale and mask; dout is the incoming gradient dO
 * (bf16, same layout rules as o); dq, dk, dv (bf16) are written. With
 * deterministic != 0 the dQ reduction runs in a fixed order and repeated calls
 * on identical inputs give bitwise-identical dq/dk/dv on the same device. This
 * implementation reduces dQ inside one query-stationary CTA per tile (no
 * atomics, no cross-CTA reduction), so deterministic == 0 reproduces bitwise
 * too; the flag is accepted for interface compatibility.
 *
 * cta_pair != 0 computes dK, dV with the two-SM kernel (wittx
 * "FlashAttention-4", section 反向传播的优化): a cluster of two CTAs runs one
 * tcgen05 MMA (cta_group::2) whose accumulator is split along the keys and whose
 * B operand is split along N, so each SM holds and reads half of every Q / dO
 * tile. Only d_qk = d_v = 128 without block lists (else ATTN_ERR_UNSUPPORTED);
 * the results are the same gradients within rounding, bitwise reproducible.
 * The default (0) is the one-SM kernel, the faster of the two on GB300: one
 * pair MMA takes ~107 cycles to issue, more than the 64 cycles of work an
 * N = 128 instruction gives each SM. */
typedef struct attn_bwd_params {
  attn_fwd_params fwd;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  int64_t do_batch_stride, do_row_stride, do_head_stride;
  int64_t dq_batch_stride, dq_row_stride, dq_head_stride;
  int64_t dk_batch_stride, dk_row_stride, dk_head_stride;
  int64_t dv_batch_stride, dv_row_stride, dv_head_stride;
  int32_t deterministic;
  int32_t cta_pair;
  /* Optional (each may be NULL): CUDA events (cudaEvent_t) recorded on the
   * stream after the D = rowsum(dO * O) pass [0], after the dK/dV kernel [1]
   * and after the dQ kernel [2], for timing the phases. */
  void* phase_events[3];
  /* single_pass != 0: the backward of wittx "FlashAttention-4", 反向传播的优化:
   * one key-stationary kernel computes dK, dV and, per 64-query step, the dQ
   * partial dS K, which it adds into an fp32 dQ buffer in the workspace
   * (red.global.add in L2); a last pass writes dQ * softmax_scale in bf16.
   * With deterministic != 0 the adds to each 64-row query tile are ordered
   * by key tile through one int32 semaphore per (batch or sequence, head,
   * tile): a key tile waits until every earlier one has added (bounded wait,
   * else ATTN_ERR_TIMEOUT from attn_get_device_status), so repeated calls
   * are bitwise identical; with deterministic == 0 the adds land in the
   * hardware's order. Only d_qk = d_v = 64, bf16 inputs, dense or varlen,
   * no block lists, no score modification, cta_pair == 0 (else
   * ATTN_ERR_UNSUPPORTED). The workspace adds, each rounded up to 256,
   * 4 x heads x query rows x 64 bytes for the fp32 dQ and, deterministic
   * only, 4 x (batch or num_seqs) x heads x ceil(max query length / 64). */
  int32_t single_pass;
} attn_bwd_params;

/* Bytes of device workspace the matching call needs (0 means none: pass NULL).
 * The forward's workspace (also for attn_fwd_varlen and attn_fwd_block_sparse)
 * holds an fp16 copy of V, made on the stream before the attention kernel: P
 * and V enter the PV product in fp16 (11 significant bits) rather than bf16,
 * which keeps O within 1e-2 of the exact result where a few keys dominate a
 * row. Its size is 256 + 2 * (keys x heads x d_v) bytes, rounded up to 256;
 * it must be 256-byte aligned. When V holds a finite value with |v| >= 65536
 * (outside fp16's range), that call computes the PV product in bf16
 * instead. A variable-length forward that builds its tile list adds, each
 * rounded up to 256, 32 x heads x (total_q / 256 + num_seqs) bytes for the
 * list and 8 x num_seqs bytes of scratch.
 * A dense forward (bf16, d_qk = d_v = 64 or 128, exp2_emu_period 0, no score
 * modification, cta_pair 0) whose batch x heads x ceil(seqlen_q / 256) query
 * blocks number at most 74 and whose keys span at least 16 blocks of 128
 * splits its keys (split-KV): s = min(148 / blocks, key blocks / 8, 32)
 * ranges of ceil(key blocks / s) blocks (then as many ranges as that needs),
 * one CTA each, each writing O and LSE over its range, merged by a second
 * kernel in range order. Its workspace then adds s x batch x heads x seqlen_q
 * x (4 x d_v + 4) bytes (the two parts each rounded up to 256). The result
 * equals the unsplit one within rounding and is the same bits on every call
 * with the same shapes. The block-sparse forward never splits.
 * The backward's workspace holds D = rowsum(dO * O): 4 x heads x query rows
 * bytes, rounded up to 256, 16-byte aligned; a variable-length backward adds
 * its tile lists, 32 x heads x (total_k / 128 + num_seqs) bytes for dK/dV
 * (none with cta_pair) and 32 x heads x (total_q / 128 + num_seqs) for dQ, and
 * 8 x num_seqs bytes of scratch, each rounded up to 256.
 * A dense two-kernel backward (bf16, single_pass 0, any supported head size,
 * with or without a score modification) whose batch x heads x
 * ceil(seqlen_q / 128) query tiles number at most 74 and whose keys span at
 * least 16 blocks of 128 splits the keys of its dQ kernel by the forward's
 * rule over those tiles: s = min(148 / tiles, key blocks / 8, 32) ranges, one
 * CTA each, each storing its fp32 dQ over its range, added in range order by a
 * second kernel (the same bits on every call; dK and dV are unchanged). The
 * size then adds s x batch x heads x seqlen_q x d_qk x 4 bytes, rounded up to
 * 256. A call given at least the size without those bytes (but less than the
 * full size) runs unsplit. The block-sparse backward never splits. */
size_t attn_fwd_workspace_size(const attn_fwd_params* p);
size_t attn_bwd_workspace_size(const attn_bwd_params* p);

/* Dense forward: O, LSE from Q, K, V. */
attn_status_t attn_fwd(const attn_fwd_params* p, void* workspace, size_t workspace_bytes, attn_stream_t stream);
/* Block-sparse forward (the FlexAttention / block-sparse variants named in
 * wittx "FlashAttention-4", section Python写GPU内核): the dense forward
 * restricted to listed key blocks. Dense layout only (cu_seqlens NULL),
 * exp2_emu_period must be 0. Query rows form blocks of 256 (block b = rows
 * 256b .. 256b+255), keys blocks of 128. Query block b attends to the key
 * blocks kv_index[b * max_kv + j] for j < kv_count[b]; every other key is
 * masked, and `causal` still applies inside the listed blocks. With
 * lists_per_head == 0 one set of lists serves every (batch, head): kv_count
 * is int32[nqb] and kv_index int32[nqb * max_kv], nqb = ceil(seqlen_q / 256).
 * With lists_per_head == 1 each (batch b, head h) has its own set, stored one
 * after another: kv_count int32[batch * heads * nqb] and kv_index
 * int32[batch * heads * nqb * max_kv], the set of (b, h) at offsets
 * (b * heads + h) * nqb and (b * heads + h) * nqb * max_kv; other values are
 * ATTN_ERR_INVALID_ARG. Both are device arrays owned by the caller, 4-byte
 * aligned, and hold fewer than 2^31 entries. Counts are
 * clamped to [0, max_kv]; indices outside [0, ceil(seqlen_k / 128)) list
 * nothing. Each key block must be listed at most once per query block: the
 * forward counts a repeated block once per listing, and the backward's result
 * for repeated blocks is undefined. Rows that see no key get O = 0,
 * LSE = -inf. Bad arguments give ATTN_ERR_INVALID_ARG before any launch.
 * The workspace is that of attn_fwd (attn_fwd_workspace_size). The gradients
 * come from attn_bwd_block_sparse. */
attn_status_t attn_fwd_block_sparse(const attn_fwd_params* p, const int32_t* kv_count, const int32_t* kv_index,
                                    int32_t max_kv, int32_t lists_per_head, void* workspace, size_t workspace_bytes,
                                    attn_stream_t stream);
/* Variable-length forward (cu_seqlens_q / cu_seqlens_k required). */
attn_status_t attn_fwd_varlen(const attn_fwd_params* p, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream);
/* Dense backward: dQ, dK, dV from Q, K, V, O, LSE, dO. */
attn_status_t attn_bwd(const attn_bwd_params* p, void* workspace, size_t workspace_bytes, attn_stream_t stream);
/* Variable-length backward. */
attn_status_t attn_bwd_varlen(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream);

/* Block-sparse backward: the gradients of attn_fwd_block_sparse for the same
 * kv_count / kv_index / max_kv / lists_per_head (same rules, blocks listed at
 * most once; dense layout only). The lists must be on the same GPU as q. The
 * key blocks' transposed lists are built on the stream into the workspace,
 * whose size is attn_bwd_block_sparse_workspace_size(p, lists_per_head)
 * (16-byte aligned). Both modes are bitwise reproducible, as for attn_bwd. */
size_t attn_bwd_block_sparse_workspace_size(const attn_bwd_params* p, int32_t lists_per_head);
attn_status_t attn_bwd_block_sparse(const attn_bwd_params* p, const int32_t* kv_count, const int32_t* kv_index,
                                    int32_t max_kv, int32_t lists_per_head, void* workspace, size_t workspace_bytes,
                                    attn_stream_t stream);

/* Backward for callers that cannot allocate device memory (an engine that
 * plans all memory up front and forbids later cudaMalloc, a plugin that is
 * handed only tensors, a loop where an allocation's possible device
 * synchronisation is unacceptable). Same computation and arguments as
 * attn_bwd / attn_bwd_varlen (chosen by whether fwd.cu_seqlens_q is NULL), but
 * no workspace: the scratch lives in a fixed array inside the library of
 * ATTN_BWD_NOALLOC_SCRATCH_BYTES bytes per GPU that loads the library, held
 * until process exit. The attention method has no counterpart to this entry
 * point; it exists only for these callers. Limit: the workspace that
 * attn_bwd would need, without the split-key dQ partials (which it uses only
 * when the array also holds them), must not exceed
 * ATTN_BWD_NOALLOC_SCRATCH_BYTES (4 bytes per batch x head x
 * query row, so up to 2,097,152 such rows dense; variable length adds the
 * tile lists), else ATTN_ERR_WORKSPACE and
 * nothing is launched. The first call on each device resolves the array's
 * address and should come before any stream capture. All calls share the one
 * array: calls that may overlap on the GPU race and must be serialised by the
 * caller. Allocates nothing (no cudaMalloc, no cudaFree). */
#define ATTN_BWD_NOALLOC_SCRATCH_BYTES (8u << 20)
attn_status_t attn_bwd_noalloc(const attn_bwd_params* p, attn_stream_t stream);

/* Diagnostic: evaluates the kernels' two exp2 paths on n device floats x:
 * y_poly = Cody-Waite split + cubic on the FMA pipe (NULL to skip),
 * y_hw = the hardware ex2 approximation (NULL to skip). Same code as the
 * forward kernel's softmax uses (wittx "FlashAttention-4", section
 * 用软件"伪造"硬件指令). */
attn_status_t attn_exp2_eval(const float* x, float* y_poly, float* y_hw, int64_t n, attn_stream_t stream);

/* Diagnostic for the failure path of the bounded waits: launches the dense
 * forward kernel (d_qk = d_v = 64, exp2_emu_period 0, seqlen_q, seqlen_k >= 1,
 * other rules as attn_fwd) in a mode where its loader issues no copies and
 * every wait gives up after spin_limit polls (1 <= spin_limit <= 2^20). The
 * MMA and softmax waits then run out: the kernel records ATTN_ERR_TIMEOUT in
 * the device status word (code 1 << 24 | the site of the first wait that gave
 * up), leaves O and LSE unspecified, and returns with no copy or MMA in
 * flight, so the context stays usable. Read the outcome with
 * attn_get_device_status. Not part of the computation; it exists to test
 * that a wait that runs out is reported instead of hanging. */
attn_status_t attn_diag_wait_timeout(const attn_fwd_params* p, uint32_t spin_limit, attn_stream_t stream);

/* Synchronises `stream`, then returns ATTN_OK if no kernel recorded a
 * failure since the last call, else ATTN_ERR_TIMEOUT (the word is cleared).
 * If detail != NULL it receives the raw status word (code << 24 | site). */
attn_status_t attn_get_device_status(attn_stream_t stream, uint32_t* detail);

/* Human-readable name of a status code (static storage). */
const char* attn_status_string(attn_status_t s);

/* Last CUDA error string seen by the library on this thread ("" if none). */
const char* attn_last_cuda_error(void);

/* ABI checks for bindings: ATTN_ABI_VERSION and sizeof of the parameter structs. */
int32_t attn_abi_version(void);
size_t attn_fwd_params_size(void);
size_t attn_bwd_params_size(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H_ */
