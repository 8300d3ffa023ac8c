/*
 * mha.h -- C ABI of libmha.so: multi-head scaled dot-product attention forward
 * on one GB300 (sm_103a).
 *
 * Operation ("Attention Is All You Need", Section 3.2.1, Equation (1)):
 *     Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 * computed independently for every sequence b in [0, B) and head h in [0, H),
 * i.e. all heads in parallel (Section 3.2.2; cookipedia article, section
 * "Transformer の構造": the n_head x d_k vector of each step is split into
 * heads, attention runs on every head, and the head outputs are concatenated).
 * For query row i of (b, h) and its visible keys j:
 *     s_j = scale * (q_i . k_j),   a_j = exp(s_j) / sum_j' exp(s_j'),
 *     o_i = sum_j a_j v_j
 * (formula page transformer-attention, section 証明).
 *
 * Masks (mask_kind):
 *   MHA_MASK_NONE         every key 0 .. Lk-1 is visible (encoder
 *                         self-attention, and cross-attention without padding).
 *   MHA_MASK_CAUSAL       key j is visible to query i only if j <= i: the
 *                         strictly-upper triangle of Q K^T is set to -inf
 *                         before the softmax, the diagonal is kept (cookipedia
 *                         article, decoder section; "Attention Is All You
 *                         Need", Section 3.1).  Requires Lq == Lk.
 *   MHA_MASK_KEY_PADDING  key j of sequence b is visible only if
 *                         j < key_lens[b] (clamped to [0, Lk]); for
 *                         cross-attention over padded encoder outputs (the
 *                         decoder's second attention layer, cookipedia
 *                         decoder section).  Not on the pages: its meaning
 *                         is this library's definition.
 *   MHA_MASK_CAUSAL_KEY_PADDING  both: key j is visible to query i of
 *                         sequence b only if j <= i and j < key_lens[b] (a
 *                         decoder's self-attention over padded sequences).
 *                         Requires Lq == Lk and key_lens.  Also this
 *                         library's definition: a key passes both masks.
 * A row with no visible key (Lk == 0, or key_lens[b] <= 0) gets output 0.
 *
 * Layout: q and out are [B, Lq, H, d_k], k and v are [B, Lk, H, d_k], dense
 * row-major (d_k fastest, then H, then L, then B).  The output therefore comes
 * out already concatenated over heads: row (b, i) holds H*d_k contiguous
 * values, ready for the output projection W^O.  d_v = d_k except in the
 * *_dv entries, where v and out rows have their own width d_v (Equation (1)
 * takes values of dimension d_v).
 *
 * Ownership: the caller owns every buffer and the stream.  No entry point
 * allocates device memory, and the device entry points never synchronise.
 * All K and V rows 0 .. Lk-1 must hold finite values: rows past a key length
 * are read (their weight is zero, but 0 * inf would still be NaN).
 *
 * Errors: argument errors are returned at once and nothing is launched.
 * Errors found on the device (a pipeline wait that timed out) are recorded in
 * a per-device status word and returned by mha_sync_status().
 */
#ifndef MHA_H
#define MHA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHA_OK = 0,
    MHA_ERR_NULL = 1,        /* a required pointer is NULL */
    MHA_ERR_SHAPE = 2,       /* negative size, causal with Lq != Lk, size overflow */
    MHA_ERR_UNSUPPORTED = 3, /* d_k not supported for this dtype, misaligned pointer, no sm_103a device */
    MHA_ERR_MASK = 4,        /* unknown mask_kind, or key_lens NULL under key padding */
    MHA_ERR_SCALE = 5,       /* scale is NaN, infinite or negative */
    MHA_ERR_LAUNCH = 6,      /* a CUDA call failed (launch, copy, synchronise) */
    MHA_ERR_TIMEOUT = 7,     /* a bounded pipeline wait on the device gave up */
    MHA_ERR_ALIAS = 8,       /* out (or lse) overlaps q, k or v (or out) */
    MHA_ERR_WORKSPACE = 9    /* workspace NULL or smaller than required */
} mha_status;

typedef enum {
    MHA_MASK_NONE = 0,
    MHA_MASK_CAUSAL = 1,
    MHA_MASK_KEY_PADDING = 2,
    MHA_MASK_CAUSAL_KEY_PADDING = 3 /* both (a bit set: causal | key padding) */
} mha_mask_kind;

/*
 * mha_fwd -- bf16 attention forward on the device.
 *   q, k, v   device pointers, bf16, layouts above; 16-byte aligned.
 *   out       device pointer, bf16 [B, Lq, H, d_k]; must not overlap q, k, v.
 *             Written with the softmax-normalised output rounded to nearest
 *             even from float32 accumulators.
 *   B, H, Lq, Lk   sizes >= 0.  B*H*Lq == 0 is a no-op returning MHA_OK;
 *             Lk == 0 writes zeros.  k and v may be NULL when Lk == 0.
 *   d_k       a multiple of 8 from 8 to 256 ("Attention Is All You Need",
 *             Section 3.2.1, fixes no width).  Heads up to 64 and up to 128
 *             run on the 64- and 128-wide kernels, which issue only the
 *             head's own ceil(d_k / 16) K steps and output columns (the
 *             tensor maps read the missing features as 0 and write only d_k
 *             columns); wider heads (to 256) run on a kernel of their own
 *             with 64-key tiles and Q held in tensor memory.
 *   mask_kind one of mha_mask_kind.
 *   key_lens  device pointer to B int32 values, read only when the mask
 *             includes key padding (may be NULL otherwise).
 *   scale     multiplier of q.k (the inverse temperature; the formula page
 *             transformer-attention, section 証明, takes the divisor tau > 0);
 *             0 selects 1/sqrt(d_k).  NaN, infinite or negative values are
 *             rejected with MHA_ERR_SCALE.
 *   stream    a cudaStream_t (NULL = the legacy default stream).
 * Products are accumulated in float32 on the tensor cores; the softmax runs in
 * float32 with exp2 and the row maximum subtracted; the probabilities are
 * rounded to bf16 before the product with V.
 * Returns MHA_OK once the work is enqueued, or an error code.
 */
int mha_fwd(const void* q, const void* k, const void* v, void* out,
            int B, int H, int Lq, int Lk, int d_k, int mask_kind,
            const int32_t* key_lens, float scale, void* stream);

/*
 * mha_fwd_f32 -- float32 attention forward on the device (all float32
 * arithmetic, CUDA cores).  Same arguments and layout as mha_fwd with float32
 * tensors (4-byte aligned); d_k from 1 to 256.
 */
int mha_fwd_f32(const void* q, const void* k, const void* v, void* out,
                int B, int H, int Lq, int Lk, int d_k, int mask_kind,
                const int32_t* key_lens, float scale, void* stream);

/*
 * mha_fwd_lse, mha_fwd_f32_lse -- mha_fwd / mha_fwd_f32 that also store, for
 * every row, the log of the softmax denominator (the log-sum-exp of the
 * row's scaled scores over its visible keys):
 *     lse[b, h, i] = log( sum_j exp(scale * q_i . k_j) )      (natural log)
 * the normaliser of Equation (1)'s softmax ("Attention Is All You Need",
 * Section 3.2.1; its exponentials are the e^{...} of the formula page
 * transformer-attention, section 証明), with a_j = exp(s_j - lse).  It is
 * what a backward pass needs to recompute the weights, and what lets partial
 * results over disjoint key ranges be merged exactly.
 *   lse   device pointer, float32 [B, H, Lq] (row i fastest), 4-byte aligned,
 *         overlapping none of q, k, v, out; must not be NULL (MHA_ERR_NULL;
 *         overlap gives MHA_ERR_ALIAS).  A row with no visible key gets -inf.
 * The value is computed in float32 from the same running maximum and sum the
 * kernel normalises the output with (before the probabilities are rounded to
 * bf16).  Other arguments, errors and behaviour as mha_fwd / mha_fwd_f32.
 */
int mha_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                int B, int H, int Lq, int Lk, int d_k, int mask_kind,
                const int32_t* key_lens, float scale, void* stream);
int mha_fwd_f32_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                    int B, int H, int Lq, int Lk, int d_k, int mask_kind,
                    const int32_t* key_lens, float scale, void* stream);

/*
 * mha_fwd_dv, mha_fwd_f32_dv -- the forward with a value width d_v of its own
 * ("Attention Is All You Need", Section 3.2.1: values of dimension d_v).
 *   q [B, Lq, H, d_k], k [B, Lk, H, d_k], v [B, Lk, H, d_v], out
 *   [B, Lq, H, d_v]; scores use the d_k columns of q and k, the output is the
 *   weighted mean of the d_v columns of v.  scale 0 selects 1/sqrt(d_k).
 *   lse   as mha_fwd_lse, or NULL for none.
 *   bf16: d_k and d_v multiples of 8 from 8 to 256 (both run on the kernel
 *   wide enough for the larger); float32: 1 to 256 each.
 * Other arguments, errors and behaviour as mha_fwd / mha_fwd_f32.
 */
int mha_fwd_dv(const void* q, const void* k, const void* v, void* out, float* lse,
               int B, int H, int Lq, int Lk, int d_k, int d_v, int mask_kind,
               const int32_t* key_lens, float scale, void* stream);
int mha_fwd_f32_dv(const void* q, const void* k, const void* v, void* out, float* lse,
                   int B, int H, int Lq, int Lk, int d_k, int d_v, int mask_kind,
                   const int32_t* key_lens, float scale, void* stream);

/*
 * mha_bwd -- gradient of mha_fwd for a loss L, given dL/dout (bf16).
 * With the row weights a_ij = exp(s_ij - lse_i) recomputed from q, k and the
 * forward's lse, g_ij = dout_i . v_j, and the formula page's derivative of
 * the weights by the scores (transformer-attention, section 証明:
 * da_j/ds_i = a_j (delta_ij - a_i)):
 *     dS_ij = a_ij (g_ij - D_i),  D_i = dout_i . out_i,
 *     dv_j = sum_i a_ij dout_i,  dk_j = scale sum_i dS_ij q_i,
 *     dq_i = scale sum_j dS_ij k_j
 * over the visible (query, key) pairs of mask_kind / key_lens; keys no query
 * sees get zero gradient.
 *   q, k, v, out  the forward's inputs and output (bf16, layouts of mha_fwd),
 *                 16-byte aligned (out is read by TMA to form D).
 *   dout          device bf16 [B, Lq, H, d_k], 16-byte aligned.
 *   lse           device float32 [B, H, Lq] from mha_fwd_lse on the same inputs.
 *   dq, dk, dv    device bf16 in the layouts of q, k, v, 16-byte aligned;
 *                 overlapping no input and each other (MHA_ERR_ALIAS).
 *   workspace     device scratch of mha_bwd_workspace_bytes(...) bytes
 *                 (D_i, float32), 16-byte aligned, owned by the caller;
 *                 overlaps no other argument (MHA_ERR_ALIAS).
 *   Other arguments as mha_fwd (d_v = d_k, any mask kind); d_k a multiple of
 *   8 from 8 to 128.
 * Products on the tensor cores in float32; the weights and dS are rounded to
 * bf16 before their products, the gradients to bf16 at the end.
 * Returns MHA_OK once enqueued, or an argument / workspace error code.
 */
int mha_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
            const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk,
            int d_k, int mask_kind, const int32_t* key_lens, float scale, void* workspace,
            size_t workspace_bytes, void* stream);

/* mha_bwd_workspace_bytes -- workspace mha_bwd needs (0 on bad sizes). */
size_t mha_bwd_workspace_bytes(int B, int H, int Lq, int Lk, int d_k);

/*
 * mha_decode -- one decode step of attention over a key/value cache, bf16.
 * At inference the decoder emits one token per step and runs again on the
 * sequence extended by it (cookipedia article, section "Transformer 全体";
 * beam search keeps four sequences going); the decoder's masked
 * self-attention then sees a usable length that grows by one per step (D2L
 * notes, the three kinds of attention, decoder layer A).  For each sequence b
 * (one per beam) and head h the step attends one query row to the first
 * cache_lens[b] cached keys and values:
 *     o[b, h] = sum_j softmax_j(scale * q[b, h] . k[b, j, h]) v[b, j, h],
 *               j < cache_lens[b]
 * -- exactly mha_fwd with Lq = 1, MHA_MASK_KEY_PADDING and key_lens =
 * cache_lens (the new token's own key and value are expected in the cache
 * already, at position cache_lens[b] - 1).
 *   q          device, bf16 [B, H, d_k] (= [B, 1, H, d_k]), 16-byte aligned.
 *   k_cache, v_cache  device, bf16 [B, Lk, H, d_k] (Lk = cache capacity),
 *              16-byte aligned; rows 0 .. Lk-1 must hold finite values.
 *   out        device, bf16 [B, H, d_k]; must not overlap q or the caches.
 *   lse        NULL, or device float32 [B, H] receiving each row's natural-log
 *              log-sum-exp (-inf when cache_lens[b] <= 0).
 *   cache_lens device int32 [B], clamped to [0, Lk]; required (MHA_ERR_MASK
 *              when NULL).  A sequence with no key gets output 0.
 *   d_k        a multiple of 8 from 8 to 256 (a head narrower than 64, 128
 *              or 256 runs on the kernel of that width with the rest of each
 *              row read as zero).  scale as in mha_fwd (0 selects 1/sqrt(d_k)).
 *   workspace  device scratch of at least mha_decode_workspace_bytes(B, H, Lk,
 *              d_k) bytes, 16-byte aligned, owned by the caller (NULL allowed
 *              when that is 0); not shared with a concurrent call.
 * Keys are split into chunks handled by separate CTAs when B*H alone would
 * leave SMs idle; the partial results (output, maximum and sum per chunk) are
 * merged exactly by a second kernel.  Products and sums are float32.
 * Returns MHA_OK once enqueued, MHA_ERR_WORKSPACE when the workspace is
 * missing or too small, or the argument codes of mha_fwd.
 */
int mha_decode(const void* q, const void* k_cache, const void* v_cache, void* out,
               float* lse, int B, int H, int Lk, int d_k, const int32_t* cache_lens,
               float scale, void* workspace, size_t workspace_bytes, void* stream);

/* mha_decode_workspace_bytes -- workspace mha_decode needs (0: none). */
size_t mha_decode_workspace_bytes(int B, int H, int Lk, int d_k);

/*
 * mha_decode_static -- mha_decode without a workspace argument: the split
 * partials go to a fixed device array inside the library (2 MiB per device,
 * mha_decode_static_scratch_bytes()), so the call allocates nothing and needs
 * no scratch from the caller.  Not from the pages: they have no counterpart;
 * it exists for callers that cannot hand over device memory.
 *   Arguments, results and errors as mha_decode; MHA_ERR_WORKSPACE when the
 *   sizes would need more than the array holds (never for any d_k the decode
 *   accepts: the split count keeps the partials under 1215 rows of at most
 *   256 + 2 floats).
 *   Nothing in the array has to start at zero: each call's split kernel
 *   writes every partial its combine kernel reads (a split that gives up on
 *   a time-out writes an empty partial, which the combine skips).
 *   Every call on a device shares the one array: calls that overlap in time
 *   (on different streams or host threads) race and give undefined results;
 *   serialise them, or use mha_decode with a workspace per stream.
 */
int mha_decode_static(const void* q, const void* k_cache, const void* v_cache, void* out,
                      float* lse, int B, int H, int Lk, int d_k, const int32_t* cache_lens,
                      float scale, void* stream);

/* mha_decode_static_scratch_bytes -- size of mha_decode_static's array. */
size_t mha_decode_static_scratch_bytes(void);

/*
 * mha_layer_fwd -- one multi-head attention layer ("Attention Is All You
 * Need", Section 3.2.2):
 *     y = MultiHead(x, m, m) = Concat(head_1, ..., head_H) W^O,
 *     head_h = Attention(x W_h^Q, m W_h^K, m W_h^V)
 * with m = x (self-attention) when mem is NULL, else the encoder memory
 * (encoder-decoder attention).  The projections run on this library's
 * tensor-core GEMM (mha_gemm_bf16: bf16 operands, float32 accumulation,
 * bf16 results); the attention is mha_fwd's kernel reading the projection
 * output in place (no transposed or split copies: the tensor maps take the
 * packed rows' stride) and writing the heads' concatenation that the W^O
 * GEMM reads.  Every kernel the layer launches is this library's.
 *   x       device bf16 [B, Lq, d_model], 16-byte aligned.
 *   mem     device bf16 [B, Lk, d_model] or NULL (then Lk must equal Lq).
 *   w_qkv   device bf16 [d_model, 3 H d_k]: W^Q, W^K, W^V side by side, head h
 *           at columns h d_k .. h d_k + d_k - 1 of each block.
 *   w_o     device bf16 [H d_k, d_model].
 *   y       device bf16 [B, Lq, d_model]; overlaps none of the others.
 *   d_model a multiple of 8; d_k as mha_fwd (a multiple of 8 up to 256);
 *           d_v = d_k.  mask_kind, key_lens, scale as mha_fwd.
 *   workspace  device, mha_layer_workspace_bytes(...) bytes, 256-byte
 *           aligned, owned by the caller (the projections and the heads'
 *           output); overlaps no argument.
 * Errors as mha_fwd, MHA_ERR_WORKSPACE for a missing or short workspace.
 * Lk == 0 writes zeros.
 */
int mha_layer_fwd(const void* x, const void* mem, const void* w_qkv, const void* w_o, void* y,
                  int B, int Lq, int Lk, int d_model, int H, int d_k, int mask_kind,
                  const int32_t* key_lens, float scale, void* workspace,
                  size_t workspace_bytes, void* stream);

/* mha_layer_workspace_bytes -- workspace mha_layer_fwd needs; 0 on bad sizes. */
size_t mha_layer_workspace_bytes(int B, int Lq, int Lk, int d_model, int H, int d_k);

/*
 * mha_gemm_bf16 -- the layer's projection product on the tensor cores
 * ("Attention Is All You Need", Section 3.2.2: Q W^Q, K W^K, V W^V and
 * Concat(heads) W^O are plain matrix products):
 *     c[M x N] = a[M x K] b[K x N]
 * all row-major bf16 in device memory, float32 accumulation, c rounded to
 * bf16 (RNE).  lda, ldb, ldc: elements between consecutive rows (>= K, N, N;
 * multiples of 8); a, b, c 16-byte aligned; c overlaps neither a nor b.
 * K == 0 writes zeros.  Returns MHA_OK once enqueued, MHA_ERR_SHAPE,
 * MHA_ERR_NULL, MHA_ERR_UNSUPPORTED (alignment) or MHA_ERR_ALIAS.
 */
int mha_gemm_bf16(const void* a, const void* b, void* c, int M, int N, int K, long long lda,
                  long long ldb, long long ldc, void* stream);

/*
 * mha_fwd_host_workspace_bytes -- device workspace mha_fwd_host needs for
 * these sizes (elem_bytes 2 for bf16, 4 for float32).  0 on bad sizes.
 */
size_t mha_fwd_host_workspace_bytes(int B, int H, int Lq, int Lk, int d_k,
                                    int elem_bytes);

/*
 * mha_fwd_host -- the same operation on HOST buffers: copies q, k, v (and
 * key_lens) into the caller's device workspace, runs mha_fwd (elem_bytes 2)
 * or mha_fwd_f32 (elem_bytes 4) there, copies the output back into out and
 * waits for the stream.  The batch goes in up to four chunks of whole
 * sequences over two internal streams, so the copies in, the kernels and the
 * copies out of consecutive chunks overlap; the internal streams start after
 * the work already queued on `stream`, which waits for them.  The first call
 * on a device creates those two streams and three events, kept for the
 * process.  Calls from several host threads at once are safe: each call
 * holds a per-device lock while it queues its work on the shared internal
 * streams, so concurrent calls run one after the other on the device (use
 * mha_fwd on streams of your own to overlap them).  Each call needs its own
 * workspace.  Host buffers should be page-locked for the copies to be
 * asynchronous.  Returns the argument check's code, MHA_ERR_WORKSPACE,
 * MHA_ERR_LAUNCH, or the device status (as mha_sync_status).
 */
int mha_fwd_host(const void* q, const void* k, const void* v, void* out,
                 int B, int H, int Lq, int Lk, int d_k, int mask_kind,
                 const int32_t* key_lens, float scale, int elem_bytes,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * mha_sync_status -- waits for the stream, then returns and clears the
 * current device's status word: MHA_OK, MHA_ERR_TIMEOUT (a kernel's bounded
 * wait gave up after about a second; its outputs are undefined), or
 * MHA_ERR_LAUNCH (the stream reported a CUDA error).
 */
int mha_sync_status(void* stream);

/*
 * mha_selftest_timeout -- launches one CTA that waits on a shared-memory
 * barrier nothing ever arrives on, using the same bounded wait as the
 * attention kernels.  The wait gives up after about a second and records
 * MHA_ERR_TIMEOUT, which the next mha_sync_status(stream) returns; the CUDA
 * context stays usable.  Exercises the device-side failure reporting without
 * a fault.  Returns MHA_OK once launched.
 */
int mha_selftest_timeout(void* stream);


/* mha_status_string -- static English text for a status code.  (The test
 * hooks of the library are declared apart, in mha_test_hooks.h.) */
const char* mha_status_string(int status);

/*
 * mha_last_launch_info -- diagnostics of the last forward call (mha_fwd*)
 * on this thread: kernels launched, grid size (CTAs), threads per CTA and
 * dynamic shared memory bytes.  Any pointer may be NULL.
 */
void mha_last_launch_info(int* kernels, int* grid, int* block, int* smem_bytes);

#ifdef __cplusplus
}
#endif

#endif /* MHA_H */
