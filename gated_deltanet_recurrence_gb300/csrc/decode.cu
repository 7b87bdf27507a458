// decode.cu -- one-token gated delta rule step on a kept fp32 state (gdn_recurrent_step).
//
// "6.6 Gated DeltaNet" 6.6.8 and "[LLM Algorithms-2] Gated DeltaNet" section 4: per (sequence,
// head) and per state row r (d_k contiguous),
//     sk_r = s_r . k,  sq_r = s_r . q,
//     delta_r = beta (v_r - alpha sk_r),
//     s_r'  = alpha s_r + delta_r k,
//     y_r   = s_r' . q = alpha sq_r + delta_r (k . q),
// which is the decay / predict / write / read sequence of the recurrence with the read folded
// into the same pass, so the state is read once and written once.
//
// HBM-bound: per (sequence, head) the kernel moves 2 * d_v * d_k * 4 bytes of state plus a few
// hundred bytes of q, k, v, y.  Layout of the work: one CTA per (sequence, head); warp w owns 16
// consecutive state rows; lane l holds d_k/32 consecutive columns of each row, so every row is
// one fully coalesced 128-bit (d_k = 128) or 64-bit (d_k = 64) access per lane.  All 16 rows are
// loaded before any arithmetic (16 x 16 B in flight per lane).  The 32 dot products of a warp
// (16 rows x {k, q}) are reduced with a transposing butterfly: 31 shuffles leave dot product j
// on lane j, instead of 5 shuffles per dot product.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRowsPerWarp = 16;

template <int EPT>
struct StateVec;
template <>
struct StateVec<4> {
    static __device__ __forceinline__ void load(const float* p, float* o) {
        float4 t = __ldcs(reinterpret_cast<const float4*>(p));
        o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* o) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(o[0], o[1], o[2], o[3]));
    }
};
template <>
struct StateVec<2> {
    static __device__ __forceinline__ void load(const float* p, float* o) {
        float2 t = __ldcs(reinterpret_cast<const float2*>(p));
        o[0] = t.x; o[1] = t.y;
    }
    static __device__ __forceinline__ void store(float* p, const float* o) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(o[0], o[1]));
    }
};

// After this, lane j holds the warp-wide sum of x[j] (32 values per lane in, 1 out).
__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
#pragma unroll
    for (int width = 16; width >= 1; width >>= 1) {
        const bool upper = (lane & width) != 0;
#pragma unroll
        for (int j = 0; j < width; ++j) {
            float send = upper ? x[j] : x[j + width];
            float keep = upper ? x[j + width] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, width);
        }
    }
    return x[0];
}

template <int D, typename TIn, bool GATE>
__global__ void __launch_bounds__(D * 2) decode_kernel(DecodeArgs a) {
    constexpr int EPT = D / 32;
    static_assert(D / kRowsPerWarp * 32 == D * 2, "one warp per 16 rows");
    __shared__ float ys[GATE ? D : 1];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long unit = blockIdx.x;  // n * H + h
    const TIn* q = static_cast<const TIn*>(a.q) + unit * D;
    const TIn* k = static_cast<const TIn*>(a.k) + unit * D;
    const TIn* v = static_cast<const TIn*>(a.v) + unit * D;
    const int r0 = warp * kRowsPerWarp;
    float* S = a.state + unit * D * D + (long)r0 * D + lane * EPT;

    // state rows first: they are the bytes that matter
    float s[kRowsPerWarp][EPT];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::load(S + (long)i * D, s[i]);

    float qv[EPT], kv[EPT];
    load_vec<EPT>(q + lane * EPT, qv);
    load_vec<EPT>(k + lane * EPT, kv);
    const float vr = lane < kRowsPerWarp ? to_f32(v[r0 + lane]) : 0.0f;
    const float alpha = expf(a.g[unit]);
    const float beta = a.beta[unit];

    float ssq = 0.f, ssk = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) { ssq += qv[e] * qv[e]; ssk += kv[e] * kv[e]; }
    ssq = warp_sum(ssq);
    ssk = warp_sum(ssk);
    const float qf = a.use_l2 ? a.scale * rsqrtf(ssq + kL2Eps) : a.scale;
    const float kf = a.use_l2 ? rsqrtf(ssk + kL2Eps) : 1.0f;
    float kq = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) { qv[e] *= qf; kv[e] *= kf; kq += kv[e] * qv[e]; }
    kq = warp_sum(kq);

    float x[32];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        float dk = 0.f, dq = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { dk += s[i][e] * kv[e]; dq += s[i][e] * qv[e]; }
        x[i] = dk;
        x[kRowsPerWarp + i] = dq;
    }
    const float t = transpose_reduce32(x, lane);  // lane<16: s_r.k of row r0+lane; else s_r.q
    const float delta = beta * (vr - alpha * t);   // meaningful on lanes < 16
    const float dsh = __shfl_sync(0xffffffffu, delta, lane & (kRowsPerWarp - 1));
    const float y = alpha * t + dsh * kq;          // meaningful on lanes >= 16

#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const float di = __shfl_sync(0xffffffffu, delta, i);
#pragma unroll
        for (int e = 0; e < EPT; ++e) s[i][e] = alpha * s[i][e] + di * kv[e];
        StateVec<EPT>::store(S + (long)i * D, s[i]);
    }

    if constexpr (!GATE) {
        if (lane >= kRowsPerWarp) store_out(a.out, unit * D + r0 + lane - kRowsPerWarp, a.out_dtype, y);
    } else {
        if (lane >= kRowsPerWarp) ys[r0 + lane - kRowsPerWarp] = y;
        __syncthreads();
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { float t2 = ys[lane * EPT + e]; ss += t2 * t2; }
        ss = warp_sum(ss);
        const float rinv = rsqrtf(ss / D + a.eps);
        if (threadIdx.x < D) {
            const int r = threadIdx.x;
            const float z = a.z[unit * D + r];
            const float w = a.w ? a.w[r] : 1.0f;
            store_out(a.out, unit * D + r, a.out_dtype, w * ys[r] * rinv * z * sigmoidf_(z));
        }
    }
}

// T tokens per sequence on a state taken from a pool by index ("6.6 Gated DeltaNet" 6.6.8 applied T
// times): the state rows stay in registers across the tokens and are written back once.  The
// per-token arithmetic is the single-step kernel's.
template <int D, typename TIn, bool GATE>
__global__ void __launch_bounds__(D * 2) decode_multi_kernel(DecodeMultiArgs a) {
    constexpr int EPT = D / 32;
    __shared__ float ys[GATE ? D : 1];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int unit = blockIdx.x;  // n * H + h
    const int n = unit / a.H, h = unit % a.H;
    const int slot = a.idx ? a.idx[n] : n;
    if (slot < 0) return;                       // padding entry: nothing to do
    if (slot >= a.num_slots) {                  // checked before any state access
        if (threadIdx.x == 0) record_error(a.err, GDN_ERR_ARG);
        return;
    }
    const int r0 = warp * kRowsPerWarp;
    float* S = a.state + ((long)slot * a.H + h) * D * D + (long)r0 * D + lane * EPT;
    float s[kRowsPerWarp][EPT];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::load(S + (long)i * D, s[i]);

    for (int t = 0; t < a.T; ++t) {
        const long tok = ((long)n * a.T + t) * a.H + h;   // [N, T, H] token index
        const TIn* q = static_cast<const TIn*>(a.q) + tok * D;
        const TIn* k = static_cast<const TIn*>(a.k) + tok * D;
        const TIn* v = static_cast<const TIn*>(a.v) + tok * D;
        float qv[EPT], kv[EPT];
        load_vec<EPT>(q + lane * EPT, qv);
        load_vec<EPT>(k + lane * EPT, kv);
        const float vr = lane < kRowsPerWarp ? to_f32(v[r0 + lane]) : 0.0f;
        const float alpha = expf(a.g[tok]);
        const float beta = a.beta[tok];
        float ssq = 0.f, ssk = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { ssq += qv[e] * qv[e]; ssk += kv[e] * kv[e]; }
        ssq = warp_sum(ssq);
        ssk = warp_sum(ssk);
        const float qf = a.use_l2 ? a.scale * rsqrtf(ssq + kL2Eps) : a.scale;
        const float kf = a.use_l2 ? rsqrtf(ssk + kL2Eps) : 1.0f;
        float kq = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { qv[e] *= qf; kv[e] *= kf; kq += kv[e] * qv[e]; }
        kq = warp_sum(kq);
        float x[32];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            float dk = 0.f, dq = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) { dk += s[i][e] * kv[e]; dq += s[i][e] * qv[e]; }
            x[i] = dk;
            x[kRowsPerWarp + i] = dq;
        }
        const float tt = transpose_reduce32(x, lane);
        const float delta = beta * (vr - alpha * tt);
        const float dsh = __shfl_sync(0xffffffffu, delta, lane & (kRowsPerWarp - 1));
        const float y = alpha * tt + dsh * kq;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float di = __shfl_sync(0xffffffffu, delta, i);
#pragma unroll
            for (int e = 0; e < EPT; ++e) s[i][e] = alpha * s[i][e] + di * kv[e];
        }
        if constexpr (!GATE) {
            if (lane >= kRowsPerWarp) store_out(a.out, tok * D + r0 + lane - kRowsPerWarp, a.out_dtype, y);
        } else {
            if (lane >= kRowsPerWarp) ys[r0 + lane - kRowsPerWarp] = y;
            __syncthreads();
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) { float t2 = ys[lane * EPT + e]; ss += t2 * t2; }
            ss = warp_sum(ss);
            const float rinv = rsqrtf(ss / D + a.eps);
            if (threadIdx.x < D) {
                const int r = threadIdx.x;
                const float z = a.z[tok * D + r];
                const float w = a.w ? a.w[r] : 1.0f;
                store_out(a.out, tok * D + r, a.out_dtype, w * ys[r] * rinv * z * sigmoidf_(z));
            }
            __syncthreads();  // ys is rewritten by the next token
        }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::store(S + (long)i * D, s[i]);
}

template <int D, typename TIn>
cudaError_t launch_multi_d(const DecodeMultiArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)((long)a.N * a.H)), block(D * 2);
    if (a.z) decode_multi_kernel<D, TIn, true><<<grid, block, 0, s>>>(a);
    else decode_multi_kernel<D, TIn, false><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)((long)a.N * a.H)), block(D * 2);
    if (a.z) decode_kernel<D, TIn, true><<<grid, block, 0, s>>>(a);
    else decode_kernel<D, TIn, false><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t s) {
    if (a.d == 128)
        return a.qkv_dtype == GDN_BF16 ? launch_multi_d<128, __nv_bfloat16>(a, s) : launch_multi_d<128, float>(a, s);
    return a.qkv_dtype == GDN_BF16 ? launch_multi_d<64, __nv_bfloat16>(a, s) : launch_multi_d<64, float>(a, s);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.d == 128) return a.qkv_dtype == GDN_BF16 ? launch_d<128, __nv_bfloat16>(a, s) : launch_d<128, float>(a, s);
    return a.qkv_dtype == GDN_BF16 ? launch_d<64, __nv_bfloat16>(a, s) : launch_d<64, float>(a, s);
}

}  // namespace gdn
