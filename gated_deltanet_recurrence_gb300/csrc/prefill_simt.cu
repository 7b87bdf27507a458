// prefill_simt.cu -- chunked prefill in fp32 CUDA-core arithmetic (gdn_chunk_fwd, exact path).
//
// Algorithm: "5. 线性注意力", "Delta Rule 的 Chunk 实现".  Per chunk of C = 64 tokens of one
// (sequence, head), with q, k L2-normalised and q scaled, gc the inclusive cumulative sum of g:
//   (1) gc, decay D_ij = exp(gc_i - gc_j) (i >= j)
//   (2) A_ij = beta_i (k_i . k_j) D_ij for j < i                     (strictly lower)
//   (3) T = (I + A)^-1 by row substitution                          (unit lower triangular)
//   (4) W = T diag(beta e^gc) K,  U = T diag(beta) V
//   (5) V_new = U - W S^T;  S <- e^{gc_last} S + V_new^T diag(e^{gc_last - gc}) K
//   (6) O = diag(e^gc) Q S^T + (Q K^T * D) V_new    (with S the state at the chunk start)
// followed, when a gate is given, by out = w * O / rms(O) * silu(z).
//
// Work layout: one CTA of 256 threads per (sequence, head), walking that sequence's chunks in
// order; the state stays in registers for the whole sequence (thread t owns state row t / TPR and
// the columns p, p + TPR, ... with p = t % TPR, TPR = 256 / d_v).  All chunk operands live in
// shared memory as fp32 with rows padded to d + 1 words (no bank conflicts in the row-broadcast
// patterns used below).  A last chunk shorter than C is masked: its missing tokens take
// k = q = v = beta = g = 0, which leaves S and the real outputs unchanged.
//
// This path keeps every product in fp32 (it is the one used for fp32 inputs, where the required
// accuracy is a relative L2 error of 1e-4); bf16 inputs are upcast exactly on load.
//
// Options handled here:
//   - grouped query/key heads: value head h reads query/key head h / (H / Hk);
//   - the short convolution ("因果卷积"): each loaded element is silu(w . (x_{t-3}, .., x_t)),
//     rounded once to the input element type, the history taken from the sequence itself or,
//     before its first token, from the input state;
//   - a decay per key channel ("6.6 Gated DeltaNet" 6.6.7), template PC: gc becomes a C x d_k
//     tile (per-channel inclusive sums), and the decays enter per element:
//       A_ij  = beta_i sum_x k_ix k_jx e^(gc_ix - gc_jx),   (Q K^T * D)_ij likewise,
//       W     = T diag(beta) (K . e^gc),   O_inter = (Q . e^gc) S^T,
//       S    <- S diag(e^gc_last) + V_new^T (K . e^(gc_last - gc)),
//     where "." scales each column x by its own factor.  Every exponent used is <= 0 (the clamp
//     only touches entries above the diagonal, which are masked), so nothing overflows.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;      // chunk size
constexpr int kThreads = 256;

template <int D>
struct SimtLayout {
    static constexpr int LD = D + 1;    // padded row stride of C x D tiles (words)
    static constexpr int LC = kC + 1;   // padded row stride of C x C tiles
    static constexpr int kTile = kC * LD;
    static constexpr int kSq = kC * LC;
    // Q, K, W, U (V, then U, then O), VN (A during steps 2-3, then V_new)
    static constexpr int oQ = 0, oK = kTile, oW = 2 * kTile, oU = 3 * kTile, oVN = 4 * kTile;
    static constexpr int oT = 5 * kTile, oAq = oT + kSq;
    static constexpr int oG = oAq + kSq;  // gc, e^gc, e^(glast-gc), beta
    static constexpr int oEL = oG + 4 * kC;  // per-channel e^(gc_last) (decay per key channel)
    static constexpr int kWords = oEL + D;
    static constexpr size_t kBytes = sizeof(float) * kWords;
};

// One raw element of q, k or v at token t (absolute index) and column x, or the carried
// convolution history when t is before the sequence start bos.
template <typename TIn>
__device__ __forceinline__ float conv_tap(const TIn* base, long stride, long t, long bos, int x,
                                          const float* hist, int c) {
    if (t >= bos) return to_f32(base[t * stride + x]);
    return hist ? hist[(long)c * 3 + 3 + (t - bos)] : 0.f;
}

template <typename TIn>
__device__ __forceinline__ float load_conv(const TIn* base, long stride, long t, long bos, int x,
                                           const float* w, const float* hist, int c) {
    const float4 wc = *reinterpret_cast<const float4*>(w + (long)c * 4);
    return round_to<TIn>(conv4_silu(wc, conv_tap(base, stride, t - 3, bos, x, hist, c),
                                    conv_tap(base, stride, t - 2, bos, x, hist, c),
                                    conv_tap(base, stride, t - 1, bos, x, hist, c),
                                    to_f32(base[t * stride + x])));
}

template <int D, typename TIn, bool PC>
__global__ void __launch_bounds__(kThreads, 1) prefill_simt_kernel(PrefillArgs a) {
    using Lay = SimtLayout<D>;
    constexpr int LD = Lay::LD, LC = Lay::LC;
    constexpr int TPR = kThreads / D;       // threads per state row
    constexpr int EPT = D / TPR;            // state columns per thread
    constexpr int RG = kThreads / D;        // row groups in the W/U step
    constexpr int RPG = kC / RG;            // rows per group

    extern __shared__ float sm[];
    float* Qs = sm + Lay::oQ;
    float* Ks = sm + Lay::oK;
    float* Ws = sm + Lay::oW;
    float* Us = sm + Lay::oU;
    float* VN = sm + Lay::oVN;
    float* Ts = sm + Lay::oT;
    float* Aq = sm + Lay::oAq;
    float* gcs = sm + Lay::oG;
    float* egc = gcs + kC;
    float* ekl = gcs + 2 * kC;
    float* bts = gcs + 3 * kC;
    float* elast = sm + Lay::oEL;
    float* G = Ws;  // per-channel gc (PC only), alive until the W step overwrites it

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int unit = blockIdx.x;
    const int n = unit / a.H, h = unit % a.H;
    long bos, eos;
    if (a.cu_seqlens) {
        bos = a.cu_seqlens[n];
        eos = a.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > a.total_T) {
            if (tid == 0) record_error(a.err, GDN_ERR_CU_SEQLENS);
            return;
        }
    } else {
        const long T = a.total_T / a.num_seqs;
        bos = (long)n * T;
        eos = bos + T;
    }
    const long tok_stride = (long)a.H * D;   // elements between consecutive tokens of v, z, out
    const long qk_stride = (long)a.Hk * D;   // ... of q and k
    const int hk = h / (a.H / a.Hk);
    const TIn* qg = static_cast<const TIn*>(a.q) + (long)hk * D;
    const TIn* kg = static_cast<const TIn*>(a.k) + (long)hk * D;
    const TIn* vg = static_cast<const TIn*>(a.v) + (long)h * D;
    const float* chist = a.conv.state_in ? a.conv.state_in + (long)n * a.conv.dim * 3 : nullptr;
    const int cq0 = hk * D, ck0 = a.Hk * D + hk * D, cv0 = 2 * a.Hk * D + h * D;

    // state row r, columns x_e = p + TPR * e
    const int r = tid / TPR, p = tid % TPR;
    float S[EPT];
    {
        const float* s0 = a.initial_state ? a.initial_state + (long)unit * D * D + (long)r * D : nullptr;
#pragma unroll
        for (int e = 0; e < EPT; ++e) S[e] = s0 ? s0[p + TPR * e] : 0.0f;
    }

    for (long c0 = bos; c0 < eos; c0 += kC) {
        const int L = (eos - c0 < kC) ? (int)(eos - c0) : kC;
        // ---- load the chunk (fp32), zero-masked beyond L ----
        for (int idx = tid; idx < kC * D; idx += kThreads) {
            const int i = idx / D, x = idx % D;
            float qv = 0.f, kv = 0.f, vv = 0.f;
            if (i < L) {
                const long t = c0 + i;
                if (a.conv.w) {
                    qv = load_conv(qg, qk_stride, t, bos, x, a.conv.w, chist, cq0 + x);
                    kv = load_conv(kg, qk_stride, t, bos, x, a.conv.w, chist, ck0 + x);
                    vv = load_conv(vg, tok_stride, t, bos, x, a.conv.w, chist, cv0 + x);
                } else {
                    qv = to_f32(qg[t * qk_stride + x]);
                    kv = to_f32(kg[t * qk_stride + x]);
                    vv = to_f32(vg[t * tok_stride + x]);
                }
            }
            Qs[i * LD + x] = qv;
            Ks[i * LD + x] = kv;
            Us[i * LD + x] = vv;
        }
        if (tid < kC) {
            const bool in = tid < L;
            gcs[tid] = (in && !PC) ? a.g[(c0 + tid) * a.H + h] : 0.f;
            bts[tid] = in ? a.beta[(c0 + tid) * a.H + h] : 0.f;
        }
        if constexpr (PC) {  // per-channel inclusive sums down the chunk, one column per thread
            for (int x = tid; x < D; x += kThreads) {
                const float* gx = a.g + (c0 * a.H + h) * (long)D + x;
                float acc = 0.f;
                for (int i = 0; i < kC; ++i) {
                    acc += i < L ? gx[(long)i * a.H * D] : 0.f;
                    G[i * LD + x] = acc;
                }
                elast[x] = expf(acc);
            }
        }
        __syncthreads();

        // ---- normalise q, k rows; cumulative log-decay ----
        for (int i = warp; i < kC; i += kThreads / 32) {
            float sq = 0.f, sk = 0.f;
            for (int x = lane; x < D; x += 32) {
                sq += Qs[i * LD + x] * Qs[i * LD + x];
                sk += Ks[i * LD + x] * Ks[i * LD + x];
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            const float qf = a.use_l2 ? a.scale * rsqrtf(sq + kL2Eps) : a.scale;
            const float kf = a.use_l2 ? rsqrtf(sk + kL2Eps) : 1.0f;
            for (int x = lane; x < D; x += 32) {
                Qs[i * LD + x] *= qf;
                Ks[i * LD + x] *= kf;
            }
        }
        if (warp == 0) {
            // inclusive scan of 64 values, two per lane
            const float g0 = gcs[2 * lane], g1 = gcs[2 * lane + 1];
            float s = g0 + g1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += t;
            }
            const float c1 = s, c0v = s - g1;
            const float glast = __shfl_sync(0xffffffffu, s, 31);  // masked tokens add 0
            gcs[2 * lane] = c0v;
            gcs[2 * lane + 1] = c1;
            egc[2 * lane] = expf(c0v);
            egc[2 * lane + 1] = expf(c1);
            ekl[2 * lane] = expf(glast - c0v);
            ekl[2 * lane + 1] = expf(glast - c1);
        }
        __syncthreads();

        // ---- A (strictly lower, into VN) and the decayed Q K^T (lower incl. diagonal) ----
        {
            const int i = tid >> 2, jp = tid & 3;
            float kk[16], qk[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) { kk[m] = 0.f; qk[m] = 0.f; }
            for (int x = 0; x < D; ++x) {
                const float ki = Ks[i * LD + x], qi = Qs[i * LD + x];
                if constexpr (PC) {
                    const float gix = G[i * LD + x];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const int j = jp + 4 * m;
                        const float kj = Ks[j * LD + x] * __expf(fminf(gix - G[j * LD + x], 0.f));
                        kk[m] += ki * kj;
                        qk[m] += qi * kj;
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const float kj = Ks[(jp + 4 * m) * LD + x];
                        kk[m] += ki * kj;
                        qk[m] += qi * kj;
                    }
                }
            }
            const float gi = gcs[i], bi = bts[i];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int j = jp + 4 * m;
                const float dec = j <= i ? (PC ? 1.f : expf(gi - gcs[j])) : 0.f;
                VN[i * LC + j] = j < i ? bi * kk[m] * dec : 0.f;
                Aq[i * LC + j] = qk[m] * dec;
                Ts[i * LC + j] = i == j ? 1.f : 0.f;
            }
        }
        __syncthreads();

        // ---- T = (I + A)^-1, row by row: T_ij = -A_ij - sum_{j<m<i} A_im T_mj ----
        for (int i = 1; i < kC; ++i) {
            const int j = tid >> 2, part = tid & 3;
            float acc = 0.f;
            if (j < i)
                for (int m = j + 1 + part; m < i; m += 4) acc += VN[i * LC + m] * Ts[m * LC + j];
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (j < i && part == 0) Ts[i * LC + j] = -VN[i * LC + j] - acc;
            __syncthreads();
        }

        // ---- W = T diag(beta e^gc) K,  U = T diag(beta) V ----
        {
            const int x = tid % D, rg = tid / D;
            float wacc[RPG], uacc[RPG];
#pragma unroll
            for (int u = 0; u < RPG; ++u) { wacc[u] = 0.f; uacc[u] = 0.f; }
            for (int j = 0; j < kC; ++j) {
                const float kb = bts[j] * (PC ? __expf(G[j * LD + x]) : egc[j]) * Ks[j * LD + x];
                const float vb = bts[j] * Us[j * LD + x];
#pragma unroll
                for (int u = 0; u < RPG; ++u) {
                    const float t = Ts[(rg * RPG + u) * LC + j];
                    wacc[u] += t * kb;
                    uacc[u] += t * vb;
                }
            }
            __syncthreads();
            if constexpr (PC) {
                // fold the per-channel decays into Q (output) and K (state update) before G,
                // which lives in the W tile, is overwritten
                for (int idx = tid; idx < kC * D; idx += kThreads) {
                    const int i = idx / D, xx = idx % D;
                    const float gc = G[i * LD + xx], gl = G[(kC - 1) * LD + xx];
                    Qs[i * LD + xx] *= __expf(gc);
                    Ks[i * LD + xx] *= __expf(gl - gc);
                }
                __syncthreads();
            }
#pragma unroll
            for (int u = 0; u < RPG; ++u) {
                Ws[(rg * RPG + u) * LD + x] = wacc[u];
                Us[(rg * RPG + u) * LD + x] = uacc[u];
            }
        }
        __syncthreads();

        // ---- serial part: V_new = U - W S^T ----
        for (int i = 0; i < kC; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) acc += Ws[i * LD + p + TPR * e] * S[e];
#pragma unroll
            for (int o = 1; o < TPR; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (p == 0) VN[i * LD + r] = Us[i * LD + r] - acc;
        }
        __syncthreads();
        // ---- O = diag(e^gc) Q S^T + (Q K^T * D) V_new, into Us ----
        for (int i = 0; i < kC; ++i) {
            float inter = 0.f, intra = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) inter += Qs[i * LD + p + TPR * e] * S[e];
            for (int j = p; j <= i; j += TPR) intra += Aq[i * LC + j] * VN[j * LD + r];
            float o = (PC ? 1.f : egc[i]) * inter + intra;
#pragma unroll
            for (int s = 1; s < TPR; s <<= 1) o += __shfl_xor_sync(0xffffffffu, o, s);
            if (p == 0) Us[i * LD + r] = o;
        }
        // ---- S <- e^{glast} S + V_new^T diag(e^{glast - gc}) K ----
        {
            const float gamma = expf(gcs[kC - 1]);
#pragma unroll
            for (int e = 0; e < EPT; ++e) S[e] *= PC ? elast[p + TPR * e] : gamma;
            for (int j = 0; j < L; ++j) {
                const float vj = VN[j * LD + r] * (PC ? 1.f : ekl[j]);
#pragma unroll
                for (int e = 0; e < EPT; ++e) S[e] += vj * Ks[j * LD + p + TPR * e];
            }
        }
        __syncthreads();

        // ---- output (gated or raw) ----
        if (a.z) {
            for (int i = warp; i < L; i += kThreads / 32) {
                float ss = 0.f;
                for (int x = lane; x < D; x += 32) ss += Us[i * LD + x] * Us[i * LD + x];
                ss = warp_sum(ss);
                const float rinv = rsqrtf(ss / D + a.eps);
                const long row = (c0 + i) * tok_stride + (long)h * D;
                for (int x = lane; x < D; x += 32) {
                    const float z = a.z[row + x];
                    const float w = a.w ? a.w[x] : 1.0f;
                    store_out(a.out, row + x, a.out_dtype, w * Us[i * LD + x] * rinv * z * sigmoidf_(z));
                }
            }
        } else {
            for (int idx = tid; idx < L * D; idx += kThreads) {
                const int i = idx / D, x = idx % D;
                store_out(a.out, (c0 + i) * tok_stride + (long)h * D + x, a.out_dtype, Us[i * LD + x]);
            }
        }
        __syncthreads();
    }

    if (a.final_state) {
        float* sf = a.final_state + (long)unit * D * D + (long)r * D;
#pragma unroll
        for (int e = 0; e < EPT; ++e) sf[p + TPR * e] = S[e];
    }
}

template <int D, typename TIn, bool PC>
cudaError_t launch_simt_pc(const PrefillArgs& a, cudaStream_t s) {
    const size_t smem = SimtLayout<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(prefill_simt_kernel<D, TIn, PC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((long)a.num_seqs * a.H);
    prefill_simt_kernel<D, TIn, PC><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_simt_d(const PrefillArgs& a, cudaStream_t s) {
    return a.g_per_channel ? launch_simt_pc<D, TIn, true>(a, s) : launch_simt_pc<D, TIn, false>(a, s);
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t s) {
    if (a.d == 128)
        return a.qkv_dtype == GDN_BF16 ? launch_simt_d<128, __nv_bfloat16>(a, s) : launch_simt_d<128, float>(a, s);
    return a.qkv_dtype == GDN_BF16 ? launch_simt_d<64, __nv_bfloat16>(a, s) : launch_simt_d<64, float>(a, s);
}

}  // namespace gdn
