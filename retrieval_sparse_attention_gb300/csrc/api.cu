// api.cu -- the C ABI declared in include/gca.h: argument validation,
// defaults, the per-device status word and kernel dispatch.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "gca.h"
#include "gca_synth.h"
#include "kernels.h"

namespace gca {

static thread_local int t_launches = 0;

namespace {

__device__ int g_status_word;           // first device-side error since the last read

constexpr int kMaxDevices = 64;
struct StatusCache {
    std::mutex mu;
    unsigned long long ctx[kMaxDevices];   // context the address was looked up in
    int* ptr[kMaxDevices];                 // device address of g_status_word
} g_status_cache;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

void resolve_ctx_fns() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
}

}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, resolve_ctx_fns);
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext c = nullptr;
    if (g_ctx_get_current(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    if (g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

int* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_cache.mu);
    const unsigned long long ctx = current_context_id();
    if (!g_status_cache.ptr[dev] || ctx == 0 || ctx != g_status_cache.ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_cache.ptr[dev] = static_cast<int*>(p);
        g_status_cache.ctx[dev] = current_context_id();   // the lookup made a context current
    }
    return g_status_cache.ptr[dev];
}

void set_launch_count(int n) { t_launches = n; }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

gca_status_t check_ptrs(std::initializer_list<const void*> ps) {
    for (const void* p : ps) {
        if (!p) return GCA_ERR_INVALID_ARG;
        if (!aligned16(p)) return GCA_ERR_INVALID_ARG;
    }
    return GCA_OK;
}

// Validate params and fill defaults.  `need_pool`: the call reads K/V.
gca_status_t make_shape(const gca_params_t* p, bool need_pool, Shape* out) {
    if (!p) return GCA_ERR_INVALID_ARG;
    Shape s{};
    s.B = p->B; s.Lq = p->Lq; s.S = p->S; s.H = p->H; s.d = p->d; s.topk = p->topk;
    s.nP = p->n_pool_chunks;
    s.dtype = p->dtype;
    s.off_by_one = p->softmax_off_by_one ? 1 : 0;
    s.include_self = p->include_self ? 1 : 0;
    if (s.B < 1 || s.S < 1 || s.H < 1 || s.d < 1 || s.Lq < s.S || s.Lq % s.S != 0)
        return GCA_ERR_INVALID_ARG;
    if (s.topk < 1) return GCA_ERR_INVALID_ARG;
    if (s.dtype != GCA_BF16 && s.dtype != GCA_F32) return GCA_ERR_INVALID_ARG;
    if (p->landmark_dim < 0) return GCA_ERR_INVALID_ARG;
    if (need_pool && s.nP < 1) return GCA_ERR_INVALID_ARG;
    s.nQ = s.Lq / s.S;
    s.D = p->landmark_dim > 0 ? p->landmark_dim : s.H * s.d;
    if (!(p->score_scale >= 0.f) || !(p->attn_scale >= 0.f)) return GCA_ERR_INVALID_ARG;
    s.score_scale = p->score_scale > 0.f ? p->score_scale : 1.0f / sqrtf((float)s.D);
    s.attn_scale = p->attn_scale > 0.f ? p->attn_scale : 1.0f / sqrtf((float)s.d);
    if (s.topk > kMaxTopk) return GCA_ERR_UNSUPPORTED;
    if (s.nQ > 16384 || s.D > 8192) return GCA_ERR_UNSUPPORTED;
    if ((double)s.B * s.Lq * s.H * s.d >= 2147483647.0 * 64) return GCA_ERR_UNSUPPORTED;
    *out = s;
    return GCA_OK;
}

// Shapes the attention kernels support: bf16 runs the tensor-core kernels
// (head dimension 32, 64 or 128; S in {64, 128}), fp32 the FFMA kernels.
gca_status_t attn_supported(const Shape& s) {
    if (s.dtype == GCA_BF16) {
        const bool dim_ok = s.d == 32 || s.d == 64 || s.d == 128;
        if (!dim_ok || (s.S != 64 && s.S != 128)) return GCA_ERR_UNSUPPORTED;
    } else {
        if ((s.d != 16 && s.d != 32 && s.d != 64) || !is_pow2(s.S) || s.S < 16 || s.S > 64)
            return GCA_ERR_UNSUPPORTED;
    }
    return GCA_OK;
}

gca_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? GCA_OK : GCA_ERR_CUDA; }

}  // namespace

void note_launches(int n) { t_launches += n; }
void reset_launches() { t_launches = 0; }

}  // namespace gca

using namespace gca;

extern "C" {

const char* gca_status_string(gca_status_t s) {
    switch (s) {
        case GCA_OK: return "GCA_OK";
        case GCA_ERR_INVALID_ARG: return "GCA_ERR_INVALID_ARG";
        case GCA_ERR_UNSUPPORTED: return "GCA_ERR_UNSUPPORTED";
        case GCA_ERR_WORKSPACE: return "GCA_ERR_WORKSPACE";
        case GCA_ERR_CUDA: return "GCA_ERR_CUDA";
        case GCA_ERR_TIMEOUT: return "GCA_ERR_TIMEOUT";
        case GCA_ERR_DEVICE_INDEX: return "GCA_ERR_DEVICE_INDEX";
    }
    return "GCA_ERR_UNKNOWN";
}

int gca_last_launch_count(void) { return t_launches; }

gca_status_t gca_get_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GCA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return GCA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return GCA_ERR_CUDA;
    }
    return static_cast<gca_status_t>(v);
}

gca_status_t gca_score_topk(const gca_params_t* params, const void* landmarks, int32_t* idx,
                            float* score, float* weight, void* stream) {
    Shape s;
    gca_status_t r = make_shape(params, false, &s);
    if (r != GCA_OK) return r;
    if ((r = check_ptrs({landmarks, idx, score, weight})) != GCA_OK) return r;
    if (sizeof(float) * ((size_t)s.D + s.nQ) > 200 * 1024) return GCA_ERR_UNSUPPORTED;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    int n = 0;
    r = from_cuda(launch_score_topk(s, landmarks, nullptr, idx, score, weight, st,
                                    static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

gca_status_t gca_score_topk_noisy(const gca_params_t* params, const void* landmarks,
                                  const float* noise, int32_t* idx, float* score, float* weight,
                                  void* stream) {
    Shape s;
    gca_status_t r = make_shape(params, false, &s);
    if (r != GCA_OK) return r;
    if ((r = check_ptrs({landmarks, noise, idx, score, weight})) != GCA_OK) return r;
    if (sizeof(float) * ((size_t)s.D + 2 * (size_t)s.nQ) > 200 * 1024) return GCA_ERR_UNSUPPORTED;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    int n = 0;
    r = from_cuda(launch_score_topk(s, landmarks, noise, idx, score, weight, st,
                                    static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

size_t gca_landmark_bwd_workspace_size(const gca_params_t* params) {
    Shape s;
    if (make_shape(params, false, &s) != GCA_OK) return 0;
    return inverse_index_bytes(s.B, s.nQ, s.nQ, s.topk);
}

gca_status_t gca_landmark_bwd(const gca_params_t* params, const void* landmarks,
                              const int32_t* idx, const float* dscore, void* dlandmarks,
                              void* workspace, size_t ws_bytes, void* stream) {
    Shape s;
    gca_status_t r = make_shape(params, false, &s);
    if (r != GCA_OK) return r;
    if ((r = check_ptrs({landmarks, idx, dscore, dlandmarks})) != GCA_OK) return r;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GCA_ERR_WORKSPACE;
    if (ws_bytes < inverse_index_bytes(s.B, s.nQ, s.nQ, s.topk)) return GCA_ERR_WORKSPACE;
    int n = 0;
    r = from_cuda(launch_landmark_bwd(s, landmarks, idx, dscore, dlandmarks, workspace,
                                      static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

gca_status_t gca_fwd(const gca_params_t* params, const void* q, const void* k, const void* v,
                     const int32_t* idx, const float* weight, void* o, float* lse, void* stream) {
    Shape s;
    gca_status_t r = make_shape(params, true, &s);
    if (r != GCA_OK) return r;
    if ((r = attn_supported(s)) != GCA_OK) return r;
    if ((r = check_ptrs({q, k, v, idx, weight, o})) != GCA_OK) return r;
    if (lse && !aligned16(lse)) return GCA_ERR_INVALID_ARG;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    int n = 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    r = from_cuda(s.dtype == GCA_BF16
                      ? launch_fwd_tc(s, q, k, v, idx, weight, o, lse, st, cs, &n)
                      : launch_fwd_simt(s, q, k, v, idx, weight, o, lse, st, cs, &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

namespace {
gca_status_t swa_check(const gca_swa_params_t* p) {
    if (!p) return GCA_ERR_INVALID_ARG;
    if (p->B < 1 || p->L < 1 || p->H < 1 || p->d < 1 || p->window < 1) return GCA_ERR_INVALID_ARG;
    if (p->dtype != GCA_BF16 && p->dtype != GCA_F32) return GCA_ERR_INVALID_ARG;
    if (!(p->attn_scale >= 0.f)) return GCA_ERR_INVALID_ARG;
    if (p->dtype != GCA_BF16 || p->d != 64) return GCA_ERR_UNSUPPORTED;
    if ((long long)p->B * p->L >= (1ll << 31) || p->H > 1024) return GCA_ERR_UNSUPPORTED;
    return GCA_OK;
}
}  // namespace

gca_status_t gca_swa_fwd(const gca_swa_params_t* params, const void* q, const void* k,
                         const void* v, void* o, float* lse, void* stream) {
    gca_status_t r = swa_check(params);
    if (r != GCA_OK) return r;
    if ((r = check_ptrs({q, k, v, o})) != GCA_OK) return r;
    if (lse && !aligned16(lse)) return GCA_ERR_INVALID_ARG;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    const float scale = params->attn_scale > 0.f ? params->attn_scale : 1.0f / sqrtf((float)params->d);
    int n = 0;
    r = from_cuda(launch_swa_fwd_tc(params->B, params->L, params->H, params->window, scale, q, k, v, o,
                                    lse, st, static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

size_t gca_swa_bwd_workspace_size(const gca_swa_params_t* params) {
    if (swa_check(params) != GCA_OK) return 0;
    return swa_bwd_workspace_bytes(params->B, params->L, params->H);
}

gca_status_t gca_swa_bwd(const gca_swa_params_t* params, const void* q, const void* k,
                         const void* v, const void* o, const float* lse, const void* dout, void* dq,
                         void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream) {
    gca_status_t r = swa_check(params);
    if (r != GCA_OK) return r;
    if ((r = check_ptrs({q, k, v, o, lse, dout, dq, dk, dv})) != GCA_OK) return r;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GCA_ERR_WORKSPACE;
    if (ws_bytes < swa_bwd_workspace_bytes(params->B, params->L, params->H)) return GCA_ERR_WORKSPACE;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    const float scale = params->attn_scale > 0.f ? params->attn_scale : 1.0f / sqrtf((float)params->d);
    int n = 0;
    r = from_cuda(launch_swa_bwd_tc(params->B, params->L, params->H, params->window, scale, q, k, v,
                                    o, lse, dout, dq, dk, dv, workspace, st,
                                    static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

size_t gca_bwd_workspace_size(const gca_params_t* params) {
    Shape s;
    if (make_shape(params, true, &s) != GCA_OK) return 0;
    return bwd_workspace_layout(s).total;
}

gca_status_t gca_bwd(const gca_params_t* params, const void* q, const void* k, const void* v,
                     const int32_t* idx, const float* weight, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, float* dscore, void* workspace,
                     size_t ws_bytes, void* stream) {
    Shape s;
    gca_status_t r = make_shape(params, true, &s);
    if (r != GCA_OK) return r;
    if ((r = attn_supported(s)) != GCA_OK) return r;
    if ((r = check_ptrs({q, k, v, idx, weight, lse, dout, dq, dk, dv, dscore})) != GCA_OK) return r;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GCA_ERR_WORKSPACE;
    if (ws_bytes < bwd_workspace_layout(s).total) return GCA_ERR_WORKSPACE;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    int n = 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    r = from_cuda(s.dtype == GCA_BF16
                      ? launch_bwd_tc(s, q, k, v, idx, weight, lse, dout, dq, dk, dv, dscore,
                                      workspace, st, cs, &n)
                      : launch_bwd_simt(s, q, k, v, idx, weight, lse, dout, dq, dk, dv, dscore,
                                        workspace, st, cs, &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

size_t gca_decode_workspace_size(int n_landmarks, int D, int topk) {
    if (n_landmarks < 1 || D < 1 || topk < 1 || topk > kMaxTopk) return 0;
    return decode_workspace_bytes(n_landmarks, topk);
}

gca_status_t gca_decode_retrieve(const void* landmarks, const void* query_landmark, int N, int D,
                                 int topk, gca_dtype_t dtype, int softmax_off_by_one,
                                 float score_scale, int32_t* idx, float* score, float* weight,
                                 void* workspace, size_t ws_bytes, void* stream) {
    if (N < 1 || D < 1 || topk < 1) return GCA_ERR_INVALID_ARG;
    if (dtype != GCA_BF16 && dtype != GCA_F32) return GCA_ERR_INVALID_ARG;
    if (!(score_scale >= 0.f)) return GCA_ERR_INVALID_ARG;
    if (topk > kMaxTopk) return GCA_ERR_UNSUPPORTED;
    const int esize = dtype == GCA_BF16 ? 2 : 4;
    if ((D * esize) % 16 != 0 || D * esize > 16 * 256) return GCA_ERR_UNSUPPORTED;
    gca_status_t r = check_ptrs({landmarks, query_landmark, idx, score, weight});
    if (r != GCA_OK) return r;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GCA_ERR_WORKSPACE;
    if (ws_bytes < decode_workspace_bytes(N, topk)) return GCA_ERR_WORKSPACE;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    const float sc = score_scale > 0.f ? score_scale : 1.0f / sqrtf((float)D);
    int n = 0;
    r = from_cuda(launch_decode_retrieve(landmarks, query_landmark, N, D, topk, dtype,
                                         softmax_off_by_one ? 1 : 0, sc, idx, score, weight,
                                         workspace, st, static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

gca_status_t gca_gather_chunks(const void* src_k, const void* src_v, int n_src,
                               size_t chunk_bytes, const int32_t* idx, int topk, void* dst_k,
                               void* dst_v, int32_t* dst_idx, void* stream) {
    if (n_src < 1 || topk < 1 || chunk_bytes == 0 || chunk_bytes % 16 != 0) return GCA_ERR_INVALID_ARG;
    if (topk > kMaxTopk) return GCA_ERR_UNSUPPORTED;
    gca_status_t r = check_ptrs({src_k, src_v, idx, dst_k, dst_v, dst_idx});
    if (r != GCA_OK) return r;
    int* st = status_word();
    if (!st) return GCA_ERR_CUDA;
    int n = 0;
    r = from_cuda(launch_gather_chunks(src_k, src_v, n_src, chunk_bytes, idx, topk, dst_k, dst_v,
                                       dst_idx, st, static_cast<cudaStream_t>(stream), &n));
    if (r == GCA_OK) t_launches = n;
    return r;
}

gca_status_t gca_synth_fill_hash(void* dst, size_t n_elems, gca_dtype_t dtype, uint64_t seed,
                                 uint64_t tensor_id, uint64_t first_elem, void* stream) {
    if (!dst || (dtype != GCA_BF16 && dtype != GCA_F32)) return GCA_ERR_INVALID_ARG;
    if (n_elems == 0) return GCA_OK;
    return from_cuda(launch_synth_fill(dst, n_elems, dtype, seed, tensor_id, first_elem,
                                       static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
