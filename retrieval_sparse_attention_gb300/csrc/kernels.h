// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gca.h"

namespace gca {

// Optional per-kernel CUDA-event bracketing (include/gca_prof.h).
void prof_begin(cudaStream_t st, const char* name);
void prof_end(cudaStream_t st);
#define GCA_LAUNCH(name, st, ...)          \
    do {                                   \
        ::gca::prof_begin((st), (name));   \
        __VA_ARGS__;                       \
        ::gca::prof_end((st));             \
    } while (0)

// Device address of the status word of the current device (looked up once
// per device and CUDA context), or nullptr if the lookup failed.
int* status_word();
// Record the launch count of the call that just succeeded, for
// gca_last_launch_count() (per host thread).
void set_launch_count(int n);
// Identity of the CUDA context current on this host thread (cuCtxGetId), or
// 0 if none is current or it cannot be read.  Per-device caches of symbol
// addresses compare it so that they are looked up again in a new context
// (after cudaDeviceReset, for instance).
unsigned long long current_context_id();

// Validated, defaulted parameters of one call.
struct Shape {
    int B, Lq, S, H, d, topk;
    int nQ;               // query chunks per row = Lq / S
    int nP;               // pool chunks per row
    int D;                // landmark dimension
    gca_dtype_t dtype;
    int off_by_one;
    int include_self;
    float score_scale;
    float attn_scale;
};

// Byte offsets of the pieces of the backward workspace.
struct BwdWorkspace {
    size_t delta_off;     // fp32 delta_t^j = dO_t . O_t^j: [B, Lq, H, topk] (FFMA path) or
                          // [B, nQ, topk, H, S] rows (tensor-core path)
    size_t dwpart_off;    // fp32 [B, nQ, H, 4, topk]: partial sums of delta over a quarter
                          // of the chunk's tokens (each quarter one TMEM lane quadrant)
    size_t lse2_off;      // fp32 [B, nQ, topk, H, S]: lse * log2(e) rows for the key pass
    size_t count_off;     // int32 [B, nP]: how many (c, j) retrieved each pool chunk
    size_t offset_off;    // int32 [B, nP + 1]: CSR offsets of the inverse index
    size_t entry_off;     // int32 [B, nQ * topk]: entries c * topk + j, ascending
    size_t entry_w_off;   // fp32 [B, nQ * topk]: the fusion weight w[b][c][j] of each entry
    size_t order_off;     // int32 [B, nP]: each row's chunks by descending retrieval count
    size_t total;
};
BwdWorkspace bwd_workspace_layout(const Shape& s);

// Decode workspace: ticket counter + per-block candidate lists.
int decode_max_blocks(int N);
size_t decode_workspace_bytes(int N, int topk);

// noise [B, nQ, nQ] fp32 or nullptr (plain top-k)
cudaError_t launch_score_topk(const Shape& s, const void* lm, const float* noise, int32_t* idx,
                              float* score, float* weight, int* status, cudaStream_t st,
                              int* launches);

// The same on the tensor cores (bf16 landmarks, D a multiple of 64, at least two chunks, k <= 16).
bool score_topk_tc_supported(const Shape& s);
cudaError_t launch_score_topk_tc(const Shape& s, const void* lm, const float* noise, int32_t* idx,
                                 float* score, float* weight, int* status, cudaStream_t st);

// Landmark gradients; ws holds an inverse index (inverse_index_bytes()).
size_t inverse_index_bytes(int B, int nQ, int nP, int topk);
cudaError_t launch_landmark_bwd(const Shape& s, const void* lm, const int32_t* idx,
                                const float* dscore, void* dlm, void* ws, cudaStream_t st,
                                int* launches);

cudaError_t launch_decode_retrieve(const void* lm, const void* ql, int N, int D, int topk,
                                   gca_dtype_t dt, int off_by_one, float score_scale,
                                   int32_t* idx, float* score, float* weight, void* ws,
                                   int* status, cudaStream_t st, int* launches);

cudaError_t launch_fwd_simt(const Shape& s, const void* q, const void* k, const void* v,
                            const int32_t* idx, const float* w, void* o, float* lse,
                            int* status, cudaStream_t st, int* launches);

cudaError_t launch_fwd_tc(const Shape& s, const void* q, const void* k, const void* v,
                          const int32_t* idx, const float* w, void* o, float* lse, int* status,
                          cudaStream_t st, int* launches);

cudaError_t launch_bwd_simt(const Shape& s, const void* q, const void* k, const void* v,
                            const int32_t* idx, const float* w, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, float* dscore,
                            void* ws, int* status, cudaStream_t st, int* launches);

cudaError_t launch_bwd_tc(const Shape& s, const void* q, const void* k, const void* v,
                          const int32_t* idx, const float* w, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, float* dscore,
                          void* ws, int* status, cudaStream_t st, int* launches);

// Shared backward pieces (inverse index, score gradient).
// (w [B, nQ, topk]: the fusion weights, copied beside the entries into the workspace)
cudaError_t launch_inverse_index(const Shape& s, const int32_t* idx, const float* w, void* ws,
                                 cudaStream_t st, int* launches);
// Inverse index into explicit buffers: count [B, nP], offset [B, nP+1], entry [B, nQ*topk],
// and, when both are given, entry_w[i] = w at entry i's (b, c, j).
cudaError_t launch_inverse_index_to(const Shape& s, const int32_t* idx, int* count, int* offset,
                                    int* entry, const float* w, float* entry_w, cudaStream_t st,
                                    int* launches);
cudaError_t launch_dscore(const Shape& s, const int32_t* idx, const float* w, void* ws,
                          float* dscore, cudaStream_t st, int* launches);

cudaError_t launch_swa_fwd_tc(int B, int L, int H, int W, float attn_scale, const void* q,
                              const void* k, const void* v, void* o, float* lse, int* status,
                              cudaStream_t st, int* launches);
size_t swa_bwd_workspace_bytes(int B, int L, int H);
cudaError_t launch_swa_bwd_tc(int B, int L, int H, int W, float attn_scale, const void* q,
                              const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, void* ws, int* status,
                              cudaStream_t st, int* launches);
cudaError_t launch_gather_chunks(const void* src_k, const void* src_v, int n_src, size_t chunk_bytes,
                                 const int32_t* idx, int topk, void* dst_k, void* dst_v,
                                 int32_t* dst_idx, int* status, cudaStream_t st, int* launches);

cudaError_t launch_synth_fill(void* dst, size_t n, gca_dtype_t dt, uint64_t seed, uint64_t tid,
                              uint64_t first, cudaStream_t st);

}  // namespace gca
