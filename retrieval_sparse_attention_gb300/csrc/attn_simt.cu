// attn_simt.cu -- fp32 FFMA kernels of the GCA forward and backward.
//
// These carry the fp32 element type (the bf16 type runs on the tensor cores,
// attn_fwd_tc.cu / attn_bwd_tc.cu); its 1e-4 tolerance rules out the tensor
// cores' reduced-precision fp32 modes.  One CTA per (query chunk,
// head, batch row) in the query-major kernels and per (pool chunk, head,
// batch row) in the key-major one; one thread per token (or per key) row.
// Every retrieved chunk's K/V (or every retrieving chunk's Q/dO) tile is
// staged in shared memory and read by all threads as broadcasts.
//
// Forward (README "Model Architecture", Eq. 2): for slot j with chunk
// kappa_j, a_s = attn_scale q_t.k_s, O_t += w_j softmax(a) V; lse_j kept.
// Backward (App. B): with p = exp(a - lse_j), G_s = dO_t.v_s and
// delta_t^j = sum_s p_s G_s (= dO_t . O_t^j):
//   da_s = w_j p_s (G_s - delta),  dq_t += attn_scale sum_s da_s k_s,
//   dk_s += attn_scale sum_t da_ts q_t,  dv_s += w_j sum_t p_ts dO_t,
//   dw_j = sum over tokens and heads of delta_t^j.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace gca {
namespace {

template <typename T, int DH>
__global__ void fwd_simt_kernel(Shape sp, const T* __restrict__ q, const T* __restrict__ k,
                                const T* __restrict__ v, const int32_t* __restrict__ idx,
                                const float* __restrict__ w, T* __restrict__ o,
                                float* __restrict__ lse, int* status) {
    extern __shared__ float sh[];
    const int S = sp.S;
    float* Ks = sh;
    float* Vs = sh + S * DH;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const size_t ld = (size_t)sp.H * DH;
    const size_t tok = (size_t)b * sp.Lq + (size_t)c * S + t;
    float qr[DH], acc[DH];
#pragma unroll
    for (int e = 0; e < DH; ++e) {
        qr[e] = to_f(q[tok * ld + (size_t)h * DH + e]);
        acc[e] = 0.f;
    }
    for (int j = 0; j < sp.topk; ++j) {
        const size_t so = ((size_t)b * sp.nQ + c) * sp.topk + j;
        const int kap = idx[so];
        float* lp = lse ? lse + (tok * sp.H + h) * sp.topk + j : nullptr;
        if (kap < 0 || kap >= sp.nP) {
            if (kap >= sp.nP && t == 0) set_status(status, GCA_ERR_DEVICE_INDEX);
            if (lp) *lp = kap < 0 ? -INFINITY : NAN;
            continue;
        }
        const float wj = w[so];
        __syncthreads();
        const size_t row0 = (size_t)b * sp.nP * S + (size_t)kap * S;
        for (int i = t; i < S * DH; i += S) {
            const int r = i / DH, e = i % DH;
            const size_t g = (row0 + r) * ld + (size_t)h * DH + e;
            Ks[i] = to_f(k[g]);
            Vs[i] = to_f(v[g]);
        }
        __syncthreads();
        float mx = -INFINITY, l = 0.f;
        for (int s = 0; s < S; ++s) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < DH; ++e) a = fmaf(qr[e], Ks[s * DH + e], a);
            a *= sp.attn_scale;
            if (a > mx) { l = l * expf(mx - a) + 1.f; mx = a; }
            else l += expf(a - mx);
        }
        const float coef = wj / l;
        for (int s = 0; s < S; ++s) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < DH; ++e) a = fmaf(qr[e], Ks[s * DH + e], a);
            const float p = expf(a * sp.attn_scale - mx) * coef;
#pragma unroll
            for (int e = 0; e < DH; ++e) acc[e] = fmaf(p, Vs[s * DH + e], acc[e]);
        }
        if (lp) *lp = mx + logf(l);
    }
#pragma unroll
    for (int e = 0; e < DH; ++e) o[tok * ld + (size_t)h * DH + e] = from_f<T>(acc[e]);
}

template <typename T, int DH>
__global__ void bwd_q_simt_kernel(Shape sp, const T* __restrict__ q, const T* __restrict__ k,
                                  const T* __restrict__ v, const int32_t* __restrict__ idx,
                                  const float* __restrict__ w, const float* __restrict__ lse,
                                  const T* __restrict__ dout, T* __restrict__ dq,
                                  float* __restrict__ delta, float* __restrict__ dwpart,
                                  int* status) {
    extern __shared__ float sh[];
    const int S = sp.S;
    float* Ks = sh;
    float* Vs = sh + S * DH;
    float* red = sh + 2 * S * DH;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const size_t ld = (size_t)sp.H * DH;
    const size_t tok = (size_t)b * sp.Lq + (size_t)c * S + t;
    float qr[DH], gr[DH], dqa[DH];
#pragma unroll
    for (int e = 0; e < DH; ++e) {
        qr[e] = to_f(q[tok * ld + (size_t)h * DH + e]);
        gr[e] = to_f(dout[tok * ld + (size_t)h * DH + e]);
        dqa[e] = 0.f;
    }
    for (int j = 0; j < sp.topk; ++j) {
        const size_t so = ((size_t)b * sp.nQ + c) * sp.topk + j;
        const int kap = idx[so];
        const size_t di = (tok * sp.H + h) * sp.topk + j;
        const size_t pi = (((size_t)b * sp.nQ + c) * sp.H + h) * 4 * sp.topk + j;   // quadrant 0
        if (kap < 0 || kap >= sp.nP) {
            if (kap >= sp.nP && t == 0) set_status(status, GCA_ERR_DEVICE_INDEX);
            delta[di] = 0.f;
            if (t < 4) dwpart[pi + t * sp.topk] = 0.f;
            continue;
        }
        const float wj = w[so];
        const float L = lse[di];
        __syncthreads();
        const size_t row0 = (size_t)b * sp.nP * S + (size_t)kap * S;
        for (int i = t; i < S * DH; i += S) {
            const int r = i / DH, e = i % DH;
            const size_t g = (row0 + r) * ld + (size_t)h * DH + e;
            Ks[i] = to_f(k[g]);
            Vs[i] = to_f(v[g]);
        }
        __syncthreads();
        float dl = 0.f;
        for (int s = 0; s < S; ++s) {
            float a = 0.f, G = 0.f;
#pragma unroll
            for (int e = 0; e < DH; ++e) {
                a = fmaf(qr[e], Ks[s * DH + e], a);
                G = fmaf(gr[e], Vs[s * DH + e], G);
            }
            dl = fmaf(expf(a * sp.attn_scale - L), G, dl);
        }
        for (int s = 0; s < S; ++s) {
            float a = 0.f, G = 0.f;
#pragma unroll
            for (int e = 0; e < DH; ++e) {
                a = fmaf(qr[e], Ks[s * DH + e], a);
                G = fmaf(gr[e], Vs[s * DH + e], G);
            }
            const float da = wj * expf(a * sp.attn_scale - L) * (G - dl) * sp.attn_scale;
#pragma unroll
            for (int e = 0; e < DH; ++e) dqa[e] = fmaf(da, Ks[s * DH + e], dqa[e]);
        }
        delta[di] = dl;
        red[t] = dl;
        __syncthreads();
        for (int o2 = S / 2; o2 > 0; o2 >>= 1) {     // fixed-order tree over the chunk
            if (t < o2) red[t] += red[t + o2];
            __syncthreads();
        }
        if (t == 0) dwpart[pi] = red[0];
        if (t > 0 && t < 4) dwpart[pi + t * sp.topk] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < DH; ++e) dq[tok * ld + (size_t)h * DH + e] = from_f<T>(dqa[e]);
}

template <typename T, int DH>
__global__ void bwd_kv_simt_kernel(Shape sp, const T* __restrict__ q, const T* __restrict__ k,
                                   const T* __restrict__ v, const float* __restrict__ w,
                                   const float* __restrict__ lse, const T* __restrict__ dout,
                                   const float* __restrict__ delta, const int* __restrict__ offset,
                                   const int* __restrict__ entry, T* __restrict__ dk,
                                   T* __restrict__ dv) {
    extern __shared__ float sh[];
    const int S = sp.S;
    float* Qs = sh;
    float* Gs = sh + S * DH;
    float* Ls = sh + 2 * S * DH;
    float* Ds = Ls + S;
    const int kap = blockIdx.x, h = blockIdx.y, b = blockIdx.z, s = threadIdx.x;
    const size_t ld = (size_t)sp.H * DH;
    const size_t krow = (size_t)b * sp.nP * S + (size_t)kap * S + s;
    float kr[DH], vr[DH], dka[DH], dva[DH];
#pragma unroll
    for (int e = 0; e < DH; ++e) {
        kr[e] = to_f(k[krow * ld + (size_t)h * DH + e]);
        vr[e] = to_f(v[krow * ld + (size_t)h * DH + e]);
        dka[e] = 0.f;
        dva[e] = 0.f;
    }
    const int nE = sp.nQ * sp.topk;
    const int* off = offset + (size_t)b * (sp.nP + 1);
    const int* ent = entry + (size_t)b * nE;
    for (int n = off[kap]; n < off[kap + 1]; ++n) {
        const int e_ = ent[n];
        const int c = e_ / sp.topk, j = e_ % sp.topk;
        const float wj = w[((size_t)b * sp.nQ + c) * sp.topk + j];
        __syncthreads();
        const size_t qrow0 = (size_t)b * sp.Lq + (size_t)c * S;
        for (int i = s; i < S * DH; i += S) {
            const int r = i / DH, e = i % DH;
            const size_t g = (qrow0 + r) * ld + (size_t)h * DH + e;
            Qs[i] = to_f(q[g]);
            Gs[i] = to_f(dout[g]);
        }
        Ls[s] = lse[((qrow0 + s) * sp.H + h) * sp.topk + j];
        Ds[s] = delta[((qrow0 + s) * sp.H + h) * sp.topk + j];
        __syncthreads();
        for (int t = 0; t < S; ++t) {
            float a = 0.f, G = 0.f;
#pragma unroll
            for (int e = 0; e < DH; ++e) {
                a = fmaf(Qs[t * DH + e], kr[e], a);
                G = fmaf(Gs[t * DH + e], vr[e], G);
            }
            const float p = expf(a * sp.attn_scale - Ls[t]);
            const float da = wj * p * (G - Ds[t]) * sp.attn_scale;
            const float pw = wj * p;
#pragma unroll
            for (int e = 0; e < DH; ++e) {
                dka[e] = fmaf(da, Qs[t * DH + e], dka[e]);
                dva[e] = fmaf(pw, Gs[t * DH + e], dva[e]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < DH; ++e) {
        dk[krow * ld + (size_t)h * DH + e] = from_f<T>(dka[e]);
        dv[krow * ld + (size_t)h * DH + e] = from_f<T>(dva[e]);
    }
}

template <typename T, int DH>
cudaError_t fwd_dh(const Shape& sp, const void* q, const void* k, const void* v,
                   const int32_t* idx, const float* w, void* o, float* lse, int* status,
                   cudaStream_t st) {
    auto kern = fwd_simt_kernel<T, DH>;
    const size_t smem = sizeof(float) * 2 * sp.S * DH;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    GCA_LAUNCH("fwd_simt", st, kern<<<dim3(sp.nQ, sp.H, sp.B), sp.S, smem, st>>>(sp, (const T*)q, (const T*)k, (const T*)v,
                                                     idx, w, (T*)o, lse, status));
    return cudaGetLastError();
}

template <typename T, int DH>
cudaError_t bwd_dh(const Shape& sp, const void* q, const void* k, const void* v,
                   const int32_t* idx, const float* w, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, void* ws, int* status, cudaStream_t st) {
    const BwdWorkspace L = bwd_workspace_layout(sp);
    char* base = static_cast<char*>(ws);
    float* delta = reinterpret_cast<float*>(base + L.delta_off);
    float* dwpart = reinterpret_cast<float*>(base + L.dwpart_off);
    const int* offset = reinterpret_cast<const int*>(base + L.offset_off);
    const int* entry = reinterpret_cast<const int*>(base + L.entry_off);
    auto kq = bwd_q_simt_kernel<T, DH>;
    const size_t smq = sizeof(float) * (2 * sp.S * DH + sp.S);
    cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
    GCA_LAUNCH("bwd_q_simt", st, kq<<<dim3(sp.nQ, sp.H, sp.B), sp.S, smq, st>>>(sp, (const T*)q, (const T*)k, (const T*)v, idx,
                                                  w, lse, (const T*)dout, (T*)dq, delta, dwpart,
                                                  status));
    auto kkv = bwd_kv_simt_kernel<T, DH>;
    const size_t smk = sizeof(float) * (2 * sp.S * DH + 2 * sp.S);
    cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
    GCA_LAUNCH("bwd_kv_simt", st, kkv<<<dim3(sp.nP, sp.H, sp.B), sp.S, smk, st>>>(sp, (const T*)q, (const T*)k, (const T*)v, w,
                                                   lse, (const T*)dout, delta, offset, entry,
                                                   (T*)dk, (T*)dv));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const Shape& sp, const void* q, const void* k, const void* v,
                            const int32_t* idx, const float* w, void* o, float* lse,
                            int* status, cudaStream_t st, int* launches) {
    cudaError_t e = cudaErrorInvalidValue;
    if (sp.dtype == GCA_F32) {
        if (sp.d == 16) e = fwd_dh<float, 16>(sp, q, k, v, idx, w, o, lse, status, st);
        if (sp.d == 32) e = fwd_dh<float, 32>(sp, q, k, v, idx, w, o, lse, status, st);
        if (sp.d == 64) e = fwd_dh<float, 64>(sp, q, k, v, idx, w, o, lse, status, st);
    }
    if (e == cudaSuccess) *launches += 1;
    return e;
}

cudaError_t launch_bwd_simt(const Shape& sp, const void* q, const void* k, const void* v,
                            const int32_t* idx, const float* w, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, float* dscore,
                            void* ws, int* status, cudaStream_t st, int* launches) {
    cudaError_t e = launch_inverse_index(sp, idx, w, ws, st, launches);
    if (e != cudaSuccess) return e;
    e = cudaErrorInvalidValue;
    if (sp.dtype == GCA_F32) {
        if (sp.d == 16) e = bwd_dh<float, 16>(sp, q, k, v, idx, w, lse, dout, dq, dk, dv, ws, status, st);
        if (sp.d == 32) e = bwd_dh<float, 32>(sp, q, k, v, idx, w, lse, dout, dq, dk, dv, ws, status, st);
        if (sp.d == 64) e = bwd_dh<float, 64>(sp, q, k, v, idx, w, lse, dout, dq, dk, dv, ws, status, st);
    }
    if (e != cudaSuccess) return e;
    *launches += 2;
    return launch_dscore(sp, idx, w, ws, dscore, st, launches);
}

}  // namespace gca
