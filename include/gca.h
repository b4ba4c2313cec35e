/*
 * gca.h -- C ABI of the Grouped Cross Attention (GCA) hot path on GB300.
 *
 * GCA is defined in "Efficient Length-Generalizable Attention via Causal
 * Retrieval for Long-Context Language Modeling" (Hu, Teng, Zhao, Wu, Tu;
 * ICML 2025, arXiv 2410.01651).  Each chunk of S tokens has one landmark
 * vector; the landmark of chunk c-1 scores earlier chunks, the top-k are
 * retrieved for chunk c, every token of chunk c attends separately to each
 * retrieved chunk (stage 1) and the per-chunk outputs are summed with the
 * softmaxed relevance scores as weights (stage 2).
 *
 * Conventions shared by every entry point
 *  - Tensor arguments are DEVICE pointers owned by the caller, except where
 *    an argument says "host".  The library allocates no memory and keeps no
 *    state except a per-device status word (see gca_get_status) and the
 *    fixed scratch array of gca_decode_retrieve_noalloc.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *    work is enqueued asynchronously on it.
 *  - The return value reports argument validation and launch errors.
 *    Errors detected on the device (a bounded wait that ran out, an index
 *    out of range) are recorded in the status word and returned by
 *    gca_get_status().  No call ever traps or aborts the GPU context.
 *  - Layouts are row-major, innermost dimension last.  Token tensors are
 *    [B, tokens, H, d]; the chunk c of a token tensor is tokens cS .. cS+S-1.
 *  - Pointers must be 16-byte aligned.
 *
 * Supported shapes (anything else returns GCA_ERR_UNSUPPORTED):
 *  - dtype GCA_BF16: d in {32, 64, 128}, S in {64, 128} (tensor-core path)
 *  - dtype GCA_F32 : d in {16, 32, 64}, S in {16, 32, 64} (fp32 FFMA path)
 *  - 1 <= topk <= 32, landmark dimension <= 8192, chunks per row <= 16384.
 */
#ifndef GCA_H_
#define GCA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GCA_OK = 0,
    GCA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    GCA_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shapes     */
    GCA_ERR_WORKSPACE = 3,     /* workspace missing or too small             */
    GCA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed          */
    GCA_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out         */
    GCA_ERR_DEVICE_INDEX = 6   /* the device saw an index outside its range  */
} gca_status_t;

typedef enum { GCA_BF16 = 0, GCA_F32 = 1 } gca_dtype_t;

typedef struct {
    int B;                  /* batch rows                                         */
    int Lq;                 /* query tokens per row; a multiple of S (nQ = Lq/S)  */
    int S;                  /* tokens per chunk                                   */
    int H;                  /* heads                                              */
    int d;                  /* head dimension                                     */
    int topk;               /* retrieved chunks per query chunk                   */
    int n_pool_chunks;      /* K/V chunks per row (nP); nQ in training            */
    int landmark_dim;       /* D of the landmark vectors; 0 means H*d             */
    gca_dtype_t dtype;      /* element type of landmarks and all token tensors    */
    int softmax_off_by_one; /* 0: vanilla softmax; 1: denominator 1 + sum         */
    int include_self;       /* 0: candidates kappa < c-1; 1: kappa <= c-1         */
    float score_scale;      /* r = score_scale * l_{c-1}.l_kappa; 0 => 1/sqrt(D)  */
    float attn_scale;       /* logits scale inside a chunk; 0 => 1/sqrt(d)        */
} gca_params_t;

/*
 * gca_score_topk -- causal relevance scoring, top-k and weight softmax.
 * Defines: the rebuttal comment "Cmt 1" (Eq. 1 with one group:
 * r = l_t^T l_k / sqrt(d)); README "Model Architecture" (the landmark of the
 * previous chunk selects the chunks for the next one); rebuttal Q4 (Eq. 3,
 * softmax off by one).
 *   landmarks [B, nC, D] (nC = Lq / S), dtype = params->dtype.
 *   For query chunk c >= 1 with landmark chunk t = c-1, the candidates are
 *   kappa < t (or kappa <= t with include_self).  s = l_t . l_kappa is
 *   accumulated in fp32 (exact for integer landmarks with |s| < 2^24).
 *   Slots are ordered by s descending, then kappa ascending.
 *   idx    [B, nC, topk] int32: retrieved chunk, -1 for an empty slot.
 *   score  [B, nC, topk] fp32: r = score_scale * s (0 for an empty slot).
 *   weight [B, nC, topk] fp32: softmax or off-by-one softmax of the valid r
 *                              (0 for an empty slot).
 */
gca_status_t gca_score_topk(const gca_params_t* params, const void* landmarks,
                            int32_t* idx, float* score, float* weight, void* stream);

/*
 * gca_score_topk_noisy -- gca_score_topk with the training-time exploration
 * of section 3.2 (Gumbel noise is added to the relevance scores before the
 * top-k selection).  The noise is drawn by the caller.
 *   noise [B, nC, nC] fp32: noise[b][c][kappa] perturbs candidate kappa of
 *   query chunk c (entries for kappa outside the candidate set are unused).
 *   The selection key is fl32(fl32(s * score_scale) + noise), rounded step
 *   by step (no fused multiply-add); ties go to the lower chunk index.
 *   score and weight are computed from the clean scores of the selected
 *   chunks, exactly as in gca_score_topk.  Other arguments as gca_score_topk.
 */
gca_status_t gca_score_topk_noisy(const gca_params_t* params, const void* landmarks,
                                  const float* noise, int32_t* idx, float* score, float* weight,
                                  void* stream);

/*
 * gca_fwd -- GCA forward: per-chunk attention (stage 1) and weighted fusion
 * (stage 2).  Defines: README "Model Architecture" (two stages), Figure 1/2,
 * Eq. 2 (the batch form of Figure 2, rebuttal W2); App. B (the forward
 * returns O and the log-sum-exp).
 *   q [B, Lq, H, d]; k, v [B, n_pool_chunks * S, H, d].
 *   idx, weight [B, nQ, topk] as written by gca_score_topk (or by the caller;
 *   entries must be -1 or in [0, n_pool_chunks)).
 *   o   [B, Lq, H, d]: O_t = sum_j weight_j * softmax(attn_scale q_t K_j^T) V_j,
 *       0 for a chunk without a valid slot.  fp32 accumulation.
 *   lse [B, Lq, H, topk] fp32 or NULL: ln sum_s exp(attn_scale q_t.k_s) per
 *       slot, -inf for an empty slot.  Required later by gca_bwd.
 */
gca_status_t gca_fwd(const gca_params_t* params, const void* q, const void* k, const void* v,
                     const int32_t* idx, const float* weight, void* o, float* lse, void* stream);

/* Bytes of device workspace gca_bwd needs for these parameters. */
size_t gca_bwd_workspace_size(const gca_params_t* params);

/*
 * gca_bwd -- gradients of GCA into Q, K, V and the relevance scores.
 * Defines: App. B backward (gradients for Q, K, V and the weights);
 * section 3 and README "Model Architecture" (the retrieval scores receive
 * gradients from the next-token loss through the fusion weights).
 *   Inputs as gca_fwd, plus lse from gca_fwd and dout [B, Lq, H, d].
 *   dq [B, Lq, H, d]; dk, dv [B, n_pool_chunks * S, H, d] are fully
 *   overwritten (chunks that no query retrieved get 0).
 *   dscore [B, nQ, topk] fp32: dLoss/dr for valid slots, 0 for empty ones.
 *   The reduction over the queries that share a retrieved chunk is done in a
 *   fixed order without atomics, so results are bitwise reproducible.
 *   workspace: device buffer of at least gca_bwd_workspace_size() bytes,
 *   256-byte aligned, owned by the caller, contents need not be initialised.
 */
gca_status_t gca_bwd(const gca_params_t* params, const void* q, const void* k, const void* v,
                     const int32_t* idx, const float* weight, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, float* dscore, void* workspace,
                     size_t ws_bytes, void* stream);

/* Bytes of device workspace gca_landmark_bwd needs. */
size_t gca_landmark_bwd_workspace_size(const gca_params_t* params);

/*
 * gca_landmark_bwd -- gradient into the landmark vectors, closing the loop
 * from the relevance-score gradient (gca_bwd's dscore) to the retriever.
 * Defines: sections 1 and 3 (the retriever learns from the next-token loss
 * through the relevance scores) with r = score_scale * l_{c-1} . l_kappa.
 *   landmarks [B, nC, D], idx [B, nC, topk] (as used in the forward),
 *   dscore [B, nC, topk] fp32 -> dlandmarks [B, nC, D] (params->dtype),
 *   fully overwritten; fp32 accumulation in a fixed order, no atomics.
 *   The selection itself is not differentiated.
 *   workspace: >= gca_landmark_bwd_workspace_size() bytes, 256-byte aligned.
 */
gca_status_t gca_landmark_bwd(const gca_params_t* params, const void* landmarks,
                              const int32_t* idx, const float* dscore, void* dlandmarks,
                              void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace gca_decode_retrieve needs. */
size_t gca_decode_workspace_size(int n_landmarks, int D, int topk);

/*
 * gca_decode_retrieve -- decode-time retrieval: one query landmark against
 * every stored landmark, top-k, softmax.  Defines: section 3.2 and 4.3 /
 * Table 3 (retrieval runs once per chunk of generated tokens).
 *   landmarks [N, D], query_landmark [D], element type `dtype`.
 *   idx/score/weight [topk] as in gca_score_topk (score desc, index asc).
 *   workspace: >= gca_decode_workspace_size() bytes, 256-byte aligned.
 */
gca_status_t gca_decode_retrieve(const void* landmarks, const void* query_landmark, int N, int D,
                                 int topk, gca_dtype_t dtype, int softmax_off_by_one,
                                 float score_scale, int32_t* idx, float* score, float* weight,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * gca_decode_retrieve_noalloc -- gca_decode_retrieve for callers that cannot
 * allocate device memory.  The paper has no counterpart: this is a usage
 * variant of the same decode retrieval, not a different operation.
 *   Some callers are handed only their input and output buffers and may not
 *   call cudaMalloc (or any allocating routine) themselves: plugin interfaces
 *   of inference engines, runtimes that plan every device byte at start-up,
 *   and latency-critical loops where an allocation's implicit device
 *   synchronisation is not acceptable.  This entry point needs no workspace
 *   argument: its scratch (a ticket counter, a score bound and the per-CTA
 *   candidate lists)
 *   lives in a file-scope device array of GCA_DECODE_STATIC_SCRATCH_BYTES
 *   bytes that every GPU loading the library holds until the process exits.
 *   Arguments, layouts and results are those of gca_decode_retrieve.
 *   Limits: the scratch holds 32768 (CTA, rank) candidates, i.e. any N with
 *   topk <= 16, or N <= 131072 with topk <= 32; larger requests return
 *   GCA_ERR_WORKSPACE and enqueue nothing.
 *   The first call on each device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   All calls on a device share the one array, which keeps the previous
 *   call's contents (counter and bound are cleared on the stream before each
 *   launch): calls whose executions overlap on the GPU (other streams, other
 *   host threads) race on it and must be serialised by the caller.
 *   Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define GCA_DECODE_STATIC_SCRATCH_BYTES (256u + 262144u)
gca_status_t gca_decode_retrieve_noalloc(const void* landmarks, const void* query_landmark, int N,
                                         int D, int topk, gca_dtype_t dtype,
                                         int softmax_off_by_one, float score_scale, int32_t* idx,
                                         float* score, float* weight, void* stream);

/*
 * gca_gather_chunks -- bring the retrieved chunks of an offloaded K/V cache
 * into a compact device pool.  Defines: section 3.2 (past chunks can be
 * offloaded to CPU memory and reloaded when retrieved) and the rebuttal's
 * offload-cost estimate (answer to Q2 of reviewer 3).
 *   src_k, src_v: caches of n_src chunks of chunk_bytes each, in memory the
 *     device can address (device memory, or page-locked host memory, whose
 *     host pointer is device-valid under unified addressing); read-only.
 *   idx [topk] int32 (device): retrieved chunks, -1 for an empty slot.
 *   dst_k, dst_v [topk, chunk_bytes] (device): chunk idx[j] is copied to
 *     slot j; empty slots are zero-filled.
 *   dst_idx [topk] int32 (device): j for a filled slot, -1 for an empty one,
 *     i.e. the idx to pass to gca_fwd together with n_pool_chunks = topk.
 *   chunk_bytes must be a multiple of 16.  An index >= n_src is reported as
 *   GCA_ERR_DEVICE_INDEX and its slot zero-filled.
 */
gca_status_t gca_gather_chunks(const void* src_k, const void* src_v, int n_src,
                               size_t chunk_bytes, const int32_t* idx, int topk, void* dst_k,
                               void* dst_v, int32_t* dst_idx, void* stream);

/*
 * Sliding-window self-attention: the fixed-size window self-attention that a
 * DRT layer runs before its GCA module.  Defines: paper summary section 1
 * (DRT combines the top-k past chunks of GCA with fixed-size sliding-window
 * self-attention) and section 4.1.2 (a 512-token window; the GCA modules are
 * appended after the attention modules).  The norm and residual between the
 * two modules are not part of this library.
 *   Token t of a row attends to the keys max(0, t - window + 1) .. t:
 *   o_t = sum_s softmax_s(attn_scale q_t . k_s) v_s per head.
 */
typedef struct {
    int B, L, H, d;       /* q, k, v, o: [B, L, H, d], d contiguous                   */
    int window;           /* W >= 1 (512 in the paper's model)                          */
    gca_dtype_t dtype;    /* element type of q/k/v/o (GCA_BF16 with d = 64 supported)   */
    float attn_scale;     /* 0 => 1/sqrt(d)                                             */
} gca_swa_params_t;

/*
 * gca_swa_fwd -- sliding-window self-attention forward.
 *   q, k, v, o [B, L, H, d] device pointers (16-byte aligned; o fully written).
 *   lse [B, L, H] fp32 or NULL: ln sum_s exp(attn_scale q_t . k_s) over the
 *   window; needed later by gca_swa_bwd.  fp32 accumulation, bf16 output.
 *   Returns GCA_ERR_UNSUPPORTED for another dtype or head dimension.
 */
gca_status_t gca_swa_fwd(const gca_swa_params_t* params, const void* q, const void* k,
                         const void* v, void* o, float* lse, void* stream);

/* Bytes of device workspace gca_swa_bwd needs. */
size_t gca_swa_bwd_workspace_size(const gca_swa_params_t* params);

/*
 * gca_swa_bwd -- gradients of the sliding-window self-attention: for an
 * upstream gradient dout, with p_ts the forward's probabilities,
 * delta_t = dout_t . o_t and ds_ts = attn_scale p_ts (dout_t . v_s - delta_t):
 *   dq_t = sum_s ds_ts k_s,  dk_s = sum_t ds_ts q_t,  dv_s = sum_t p_ts dout_t.
 *   q, k, v, o, dout, dq, dk, dv [B, L, H, d]; lse [B, L, H] from gca_swa_fwd.
 *   dq, dk, dv are fully overwritten; fp32 accumulation in a fixed order,
 *   no atomics (bitwise reproducible).
 *   workspace: >= gca_swa_bwd_workspace_size() bytes, 256-byte aligned.
 */
gca_status_t gca_swa_bwd(const gca_swa_params_t* params, const void* q, const void* k,
                         const void* v, const void* o, const float* lse, const void* dout, void* dq,
                         void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream);

/*
 * gca_get_status -- synchronise `stream`, then return and clear the device
 * status word of the current device (GCA_OK if no device-side error was
 * recorded since the last call).
 */
gca_status_t gca_get_status(void* stream);

/* Human-readable name of a status code (static storage). */
const char* gca_status_string(gca_status_t status);

/* Number of kernel launches the most recent successful call on this host
 * thread enqueued (for launch accounting in benchmarks). */
int gca_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GCA_H_ */
