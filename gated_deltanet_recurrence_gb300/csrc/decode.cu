// decode.cu -- gated delta rule decode on kept fp32 states (gdn_recurrent_step and
// gdn_recurrent_multi_step: T tokens per sequence from a state pool, token by token in
// decode_kernel or, for several tokens, in blocks of four in the chunked form in
// decode_block_kernel).
//
// "6.6 Gated DeltaNet" 6.6.8 and "[LLM Algorithms-2] Gated DeltaNet" section 4: per (sequence,
// head) and per state row r (d_k contiguous), with alpha one value or one per key channel,
//     sk_r = s_r . (alpha k),  sq_r = s_r . (alpha q),
//     delta_r = beta (v_r - sk_r),
//     s_r'  = alpha . s_r + delta_r k,
//     y_r   = s_r' . q = sq_r + delta_r (k . q),
// which is the decay / predict / write / read sequence of the recurrence with the read folded
// into the same pass, so the state is read once and written once.
//
// HBM-bound: per (sequence, head) the kernel moves 2 * d_v * d_k * 4 bytes of state plus a few
// hundred bytes of q, k, v, y per token.  Layout of the work: one CTA per (sequence, head); warp
// w owns 16 consecutive state rows; lane l holds d_k/32 consecutive columns of each row, so every
// row is one fully coalesced 128-bit (d_k = 128) or 64-bit (d_k = 64) access per lane.  All 16
// rows are loaded before any arithmetic (16 x 16 B in flight per lane).  The 32 dot products of
// a warp (16 rows x {k, q}) are reduced with a transposing butterfly: 31 shuffles leave dot
// product j on lane j, instead of 5 shuffles per dot product.
#include <stdlib.h>

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

// The raw per-token inputs one lane needs: its q and k columns, the value of its state row, the
// decay (its key channels' logits, or the head's in g[0]), beta, and, for threads below D, the gate
// input of output channel threadIdx.x.
template <int EPT>
struct TokenInputs {
    float q[EPT], k[EPT], g[EPT], v, beta, z;
};

template <int D, typename TIn, bool GATE, bool QKV = true>
__device__ __forceinline__ TokenInputs<D / 32> load_token(const DecodeArgs& a, long tok, int h, int hk, int lane,
                                                          int vrow) {
    constexpr int EPT = D / 32;
    TokenInputs<EPT> in;
    const long vt = tok * a.H + h;      // [.., H] row of this value head
    const long qt = tok * a.Hk + hk;    // [.., Hk] row of its query/key head
    if constexpr (QKV) {  // (with the convolution, the channel owners load the raw inputs instead)
        load_vec<EPT>(static_cast<const TIn*>(a.q) + qt * D + lane * EPT, in.q);
        load_vec<EPT>(static_cast<const TIn*>(a.k) + qt * D + lane * EPT, in.k);
        in.v = to_f32(static_cast<const TIn*>(a.v)[vt * D + vrow]);
    }
    if (a.g_per_channel) load_vec<EPT>(a.g + vt * D + lane * EPT, in.g);
    else in.g[0] = a.g[vt];
    in.beta = a.beta[vt];
    in.z = GATE && threadIdx.x < D ? a.z[vt * D + threadIdx.x] : 0.f;
    return in;
}

// One CTA per (sequence, value head).  The state comes from slot idx[n] of the pool (slot n when
// idx is null), stays in registers for the T tokens, and is written back once.  Per token:
//     x' = silu(conv(x)) for x in q, k, v        (optional short convolution)
//     q, k normalised, q scaled;  qa = alpha . q, ka = alpha . k  (alpha per key channel or one
//     value for the head; alpha s . k = s . (alpha k))
//     sk_r = s_r . ka,  sq_r = s_r . qa,  delta_r = beta (v_r - sk_r)
//     s_r <- alpha . s_r + delta_r k,     y_r = sq_r + delta_r (k . q)
// The T tokens of one (sequence n, value head h) unit on this warp's 16 state rows `s` (this lane's
// columns, kept in registers); `ys` is D floats of shared memory (gate only), `cx` 3 D floats
// (convolution only).  Called by every thread of the CTA: it synchronises the CTA when a gate or
// a convolution is applied.
//
// The convolution runs once per CTA and token: each thread owns one or two of the 3 D (q | k | v,
// channel) items, keeps their three previous raw inputs in registers, convolves the token's raw
// input and writes the result to `cx`, from which every lane takes its q, k columns and v row.
template <int D, typename TIn, bool GATE, bool CONV>
__device__ __forceinline__ void decode_tokens(float (&s)[kRowsPerWarp][D / 32], const DecodeArgs& a, int n, int h,
                                              int slot, float* ys, float* cx) {
    constexpr int EPT = D / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = a.H / a.Hk, hk = h / grp;   // value head h reads query/key head h / grp
    const int r0 = warp * kRowsPerWarp;
    const int vrow = r0 + (lane & (kRowsPerWarp - 1));

    // convolution items owned by this thread: item = tid + u * blockDim (u = 0, 1), group item / D
    // (0: q, 1: k, 2: v), channel item % D; their three previous raw inputs, oldest first
    constexpr int kItems = 3 * D, kOwn = (kItems + 2 * D - 1) / (2 * D);
    const float4* w4 = reinterpret_cast<const float4*>(a.conv.w);
    float hist[CONV ? kOwn : 1][3];
    int chan[CONV ? kOwn : 1];
    if constexpr (CONV) {
        const float* si = a.conv.state_in ? a.conv.state_in + (long)slot * a.conv.dim * 3 : nullptr;
#pragma unroll
        for (int u = 0; u < kOwn; ++u) {
            const int item = threadIdx.x + u * blockDim.x, gq = item / D, c = item % D;
            chan[u] = gq == 0 ? hk * D + c : (gq == 1 ? a.Hk * D + hk * D + c : 2 * a.Hk * D + h * D + c);
#pragma unroll
            for (int j = 0; j < 3; ++j) hist[u][j] = (item < kItems && si) ? si[(long)chan[u] * 3 + j] : 0.f;
        }
    }

    // Without the convolution the raw inputs of token t + 1 are loaded while token t computes, so
    // only the first token's loads sit on the chain of a multi-token unit.  The convolution's
    // history already fills the register budget: there each token loads its own inputs.
    constexpr bool kPrefetch = !CONV;
    TokenInputs<EPT> nxt;
    if constexpr (kPrefetch) nxt = load_token<D, TIn, GATE>(a, (long)n * a.T, h, hk, lane, vrow);
    (void)w4;
    for (int t = 0; t < a.T; ++t) {
        const long tok = (long)n * a.T + t;
        const long vt = tok * a.H + h;          // [.., H] row of this value head
        TokenInputs<EPT> cur;
        if constexpr (kPrefetch) {
            cur = nxt;
            if (t + 1 < a.T) nxt = load_token<D, TIn, GATE>(a, tok + 1, h, hk, lane, vrow);
        } else {
            cur = load_token<D, TIn, GATE, false>(a, tok, h, hk, lane, vrow);
        }
        float qv[EPT], kv[EPT], alpha[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) { qv[e] = cur.q[e]; kv[e] = cur.k[e]; }
        float vr = cur.v;
        if constexpr (CONV) {
            if (t > 0) __syncthreads();  // every lane has read the previous token's cx
#pragma unroll
            for (int u = 0; u < kOwn; ++u) {
                const int item = threadIdx.x + u * blockDim.x;
                if (item < kItems) {
                    const int gq = item / D, c = item % D;
                    const TIn* src = gq == 0 ? static_cast<const TIn*>(a.q) + (tok * a.Hk + hk) * D
                                   : (gq == 1 ? static_cast<const TIn*>(a.k) + (tok * a.Hk + hk) * D
                                              : static_cast<const TIn*>(a.v) + vt * D);
                    const float x = to_f32(src[c]);
                    cx[item] = round_to<TIn>(conv4_silu(__ldg(w4 + chan[u]), hist[u][0], hist[u][1], hist[u][2], x));
                    hist[u][0] = hist[u][1];
                    hist[u][1] = hist[u][2];
                    hist[u][2] = x;
                }
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                qv[e] = cx[lane * EPT + e];
                kv[e] = cx[D + lane * EPT + e];
            }
            vr = cx[2 * D + vrow];
        }
        if (a.g_per_channel) {
#pragma unroll
            for (int e = 0; e < EPT; ++e) alpha[e] = expf(cur.g[e]);
        } else {
            const float a0 = expf(cur.g[0]);
#pragma unroll
            for (int e = 0; e < EPT; ++e) alpha[e] = a0;
        }
        const float beta = cur.beta;

        float ssq = 0.f, ssk = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { ssq += qv[e] * qv[e]; ssk += kv[e] * kv[e]; }
        ssq = warp_sum(ssq);
        ssk = warp_sum(ssk);
        const float qf = a.use_l2 ? a.scale * rsqrtf(ssq + kL2Eps) : a.scale;
        const float kf = a.use_l2 ? rsqrtf(ssk + kL2Eps) : 1.0f;
        float kq = 0.f, qa[EPT], ka[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            qv[e] *= qf;
            kv[e] *= kf;
            kq += kv[e] * qv[e];
            qa[e] = alpha[e] * qv[e];
            ka[e] = alpha[e] * kv[e];
        }
        kq = warp_sum(kq);

        // the row dot products and the update run on column pairs with the packed two-wide fp32
        // FMA / multiply (half the instructions); a dot product adds its two pair sums at the end
        float x[32];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            float2 pk = make_float2(0.f, 0.f), pq = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EPT; e += 2) {
                const float2 sv = make_float2(s[i][e], s[i][e + 1]);
                pk = __ffma2_rn(sv, make_float2(ka[e], ka[e + 1]), pk);
                pq = __ffma2_rn(sv, make_float2(qa[e], qa[e + 1]), pq);
            }
            x[i] = pk.x + pk.y;
            x[kRowsPerWarp + i] = pq.x + pq.y;
        }
        const float tt = transpose_reduce32(x, lane);  // lane < 16: s_r . ka of row r0 + lane; else s_r . qa
        const float delta = beta * (vr - tt);           // meaningful on lanes < 16
        const float dsh = __shfl_sync(0xffffffffu, delta, lane & (kRowsPerWarp - 1));
        const float y = tt + dsh * kq;                  // meaningful on lanes >= 16
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float di = __shfl_sync(0xffffffffu, delta, i);
#pragma unroll
            for (int e = 0; e < EPT; e += 2) {
                const float2 t = __fmul2_rn(make_float2(alpha[e], alpha[e + 1]), make_float2(s[i][e], s[i][e + 1]));
                const float2 r = __ffma2_rn(make_float2(di, di), make_float2(kv[e], kv[e + 1]), t);
                s[i][e] = r.x;
                s[i][e + 1] = r.y;
            }
        }

        if constexpr (!GATE) {
            if (lane >= kRowsPerWarp) store_out(a.out, vt * D + vrow, a.out_dtype, y);
        } else {
            if (lane >= kRowsPerWarp) ys[vrow] = y;
            __syncthreads();
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) { float t2 = ys[lane * EPT + e]; ss += t2 * t2; }
            ss = warp_sum(ss);
            const float rinv = rsqrtf(ss / D + a.eps);
            if (threadIdx.x < D) {
                const int r = threadIdx.x;
                const float z = cur.z;
                const float w = a.w ? a.w[r] : 1.0f;
                store_out(a.out, vt * D + r, a.out_dtype, w * ys[r] * rinv * z * sigmoidf_(z));
            }
            __syncthreads();  // ys is rewritten by the next token
        }
    }
    if constexpr (CONV) {
        // the final history of the owned items (each thread read its own items' input history
        // before the loop; with grouped heads the query/key items are written by one value head)
        if (a.conv.state_out) {
            float* so = a.conv.state_out + (long)slot * a.conv.dim * 3;
#pragma unroll
            for (int u = 0; u < kOwn; ++u) {
                const int item = threadIdx.x + u * blockDim.x;
                if (item < kItems && (item >= 2 * D || h % grp == 0))
#pragma unroll
                    for (int j = 0; j < 3; ++j) so[(long)chan[u] * 3 + j] = hist[u][j];
            }
        }
    }
}

// One CTA per (sequence, value head): the state rows are loaded into registers first (they are
// the bytes that matter), the tokens run, and the state is written back once.
template <int D, typename TIn, bool GATE, bool CONV>
__global__ void __launch_bounds__(D * 2, 2) decode_kernel(DecodeArgs a) {
    constexpr int EPT = D / 32;
    static_assert(D / kRowsPerWarp * 32 == D * 2, "one warp per 16 rows");
    __shared__ float ys[GATE ? D : 1];
    __shared__ float cx[CONV ? 3 * D : 1];
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
    float* S = a.state + ((long)slot * a.H + h) * D * D + (long)(warp * kRowsPerWarp) * D + lane * EPT;
    float s[kRowsPerWarp][EPT];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::load(S + (long)i * D, s[i]);
    decode_tokens<D, TIn, GATE, CONV>(s, a, n, h, slot, ys, cx);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::store(S + (long)i * D, s[i]);
}

// ---- several tokens per unit: blocks of kBlk tokens in the chunked form ------------------------
//
// "[LLM Algorithms-2] Gated DeltaNet" section 4 (the chunk form of the same recurrence) applied to
// a block of kBlk tokens of one unit, with S_0 the state before the block and, per key channel c,
// G_t[c] the block's cumulative log decay up to token t (one value for all channels when the decay
// is per head):
//     A[i][j] = beta_i sum_c k_i[c] k_j[c] e^(G_i - G_j)[c]   (j < i),   T = (I + A)^-1
//     W_i = sum_j T[i][j] beta_j (e^G_j . k_j),    U[i][r] = sum_j T[i][j] beta_j v_j[r]
//     V_new[i][r] = U[i][r] - s_r . W_i                       (s_r: state row r of S_0)
//     y_i[r] = s_r . (e^G_i . q_i) + sum_(j <= i) M[i][j] V_new[j][r],
//              M[i][j] = sum_c q_i[c] k_j[c] e^(G_i - G_j)[c]
//     s_r <- e^G_last . s_r + sum_j V_new[j][r] (e^(G_last - G_j) . k_j)
// which is the token-by-token update (prediction from the decayed state, write, read) regrouped,
// so a unit's tokens share one pass over its state: the 2 kBlk dot products of a state row are
// independent, and the update costs kBlk + 1 operations per element instead of 2 kBlk.  Every
// exponent is <= 0.  A block past the last token is padded with tokens that change nothing
// (k = q = v = 0, beta = 0, no decay), so any T works.
constexpr int kBlk = 4;

template <int D, typename TIn, bool GATE, bool CONV>
__global__ void __launch_bounds__(D * 2, 2) decode_block_kernel(DecodeArgs a) {
    constexpr int EPT = D / 32, NW = D / kRowsPerWarp;
    static_assert(NW >= kBlk, "one warp per token of a block");
    __shared__ __align__(16) float kn[kBlk][D];   // normalised k (then unused rows of W scratch)
    __shared__ __align__(16) float qn[kBlk][D];   // scaled, normalised q
    __shared__ __align__(16) float vv[kBlk][D];   // v
    __shared__ __align__(16) float Gs[kBlk][D];   // log decay, then its cumulative sum over the block
    __shared__ __align__(16) float Wm[kBlk][D];   // e^G_j . k_j, then W_i
    __shared__ __align__(16) float Qd[kBlk][D];   // e^G_i . q_i
    __shared__ __align__(16) float Kd[kBlk][D];   // e^(G_last - G_j) . k_j
    __shared__ __align__(16) float gL[D];         // e^G_last
    __shared__ __align__(16) float zz[GATE ? kBlk : 1][GATE ? D : 1];
    __shared__ float part[GATE ? kBlk : 1][NW];  // per warp: sum of y^2 over its 16 rows
    __shared__ float bet[kBlk], Am[kBlk][kBlk], Mm[kBlk][kBlk], Uc[kBlk][kBlk];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int unit = blockIdx.x;  // n * H + h
    const int n = unit / a.H, h = unit % a.H;
    const int grp = a.H / a.Hk, hk = h / grp;
    const int slot = a.idx ? a.idx[n] : n;
    if (slot < 0) return;
    if (slot >= a.num_slots) {
        if (tid == 0) record_error(a.err, GDN_ERR_ARG);
        return;
    }
    const int r0 = warp * kRowsPerWarp;
    float* S = a.state + ((long)slot * a.H + h) * D * D + (long)r0 * D + lane * EPT;
    float s[kRowsPerWarp][EPT];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::load(S + (long)i * D, s[i]);

    const int c0 = lane * EPT;                       // this lane's key / value channels
    const int cq = hk * D + c0, ck = a.Hk * D + cq, cv = 2 * a.Hk * D + h * D + c0;  // conv channels
    const float* cs_in = CONV && a.conv.state_in ? a.conv.state_in + (long)slot * a.conv.dim * 3 : nullptr;
    const int vrow = r0 + (lane & (kRowsPerWarp - 1));

    for (int t0 = 0; t0 < a.T; t0 += kBlk) {
        // ---- per token (warp w <- token t0 + w): inputs, convolution, norms ----
        if (warp < kBlk) {
            const int t = t0 + warp;
            float qv[EPT], kv[EPT], vx[EPT], gv[EPT], zv[EPT];
            float bt = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) { qv[e] = kv[e] = vx[e] = gv[e] = zv[e] = 0.f; }
            if (t < a.T) {
                const long tok = (long)n * a.T + t, vt = tok * a.H + h, qt = tok * a.Hk + hk;
                load_vec<EPT>(static_cast<const TIn*>(a.q) + qt * D + c0, qv);
                load_vec<EPT>(static_cast<const TIn*>(a.k) + qt * D + c0, kv);
                load_vec<EPT>(static_cast<const TIn*>(a.v) + vt * D + c0, vx);
                if constexpr (CONV) {
                    // raw inputs of tokens t-3 .. t-1: earlier tokens of this call, else the history
                    const float4* w4 = reinterpret_cast<const float4*>(a.conv.w);
                    float hq[3][EPT], hkk[3][EPT], hv[3][EPT];
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        const int tau = t - 3 + j;
                        if (tau >= 0) {
                            const long tk = (long)n * a.T + tau;
                            load_vec<EPT>(static_cast<const TIn*>(a.q) + (tk * a.Hk + hk) * D + c0, hq[j]);
                            load_vec<EPT>(static_cast<const TIn*>(a.k) + (tk * a.Hk + hk) * D + c0, hkk[j]);
                            load_vec<EPT>(static_cast<const TIn*>(a.v) + (tk * a.H + h) * D + c0, hv[j]);
                        } else {
#pragma unroll
                            for (int e = 0; e < EPT; ++e) {
                                hq[j][e] = cs_in ? cs_in[(long)(cq + e) * 3 + 3 + tau] : 0.f;
                                hkk[j][e] = cs_in ? cs_in[(long)(ck + e) * 3 + 3 + tau] : 0.f;
                                hv[j][e] = cs_in ? cs_in[(long)(cv + e) * 3 + 3 + tau] : 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < EPT; ++e) {
                        qv[e] = round_to<TIn>(conv4_silu(__ldg(w4 + cq + e), hq[0][e], hq[1][e], hq[2][e], qv[e]));
                        kv[e] = round_to<TIn>(conv4_silu(__ldg(w4 + ck + e), hkk[0][e], hkk[1][e], hkk[2][e], kv[e]));
                        vx[e] = round_to<TIn>(conv4_silu(__ldg(w4 + cv + e), hv[0][e], hv[1][e], hv[2][e], vx[e]));
                    }
                }
                if (a.g_per_channel) {
                    load_vec<EPT>(a.g + vt * D + c0, gv);
                } else {
                    const float g0 = a.g[vt];
#pragma unroll
                    for (int e = 0; e < EPT; ++e) gv[e] = g0;
                }
                bt = a.beta[vt];
                if constexpr (GATE) load_vec<EPT>(a.z + vt * D + c0, zv);
                float ssq = 0.f, ssk = 0.f;
#pragma unroll
                for (int e = 0; e < EPT; ++e) { ssq += qv[e] * qv[e]; ssk += kv[e] * kv[e]; }
                ssq = warp_sum(ssq);
                ssk = warp_sum(ssk);
                const float qf = a.use_l2 ? a.scale * rsqrtf(ssq + kL2Eps) : a.scale;
                const float kf = a.use_l2 ? rsqrtf(ssk + kL2Eps) : 1.0f;
#pragma unroll
                for (int e = 0; e < EPT; ++e) { qv[e] *= qf; kv[e] *= kf; }
            }
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                qn[warp][c0 + e] = qv[e];
                kn[warp][c0 + e] = kv[e];
                vv[warp][c0 + e] = vx[e];
                Gs[warp][c0 + e] = gv[e];
                if constexpr (GATE) zz[warp][c0 + e] = zv[e];
            }
            if (lane == 0) bet[warp] = bt;
        }
        __syncthreads();
        // ---- cumulative log decay and the decayed operand rows (one thread per channel) ----
        if (tid < D) {
            const int c = tid;
            float G[kBlk];
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kBlk; ++j) { acc += Gs[j][c]; G[j] = acc; Gs[j][c] = acc; }
            gL[c] = __expf(G[kBlk - 1]);  // every exponent here is <= 0
#pragma unroll
            for (int j = 0; j < kBlk; ++j) {
                const float eg = __expf(G[j]);
                Wm[j][c] = eg * kn[j][c];
                Qd[j][c] = eg * qn[j][c];
                Kd[j][c] = __expf(G[kBlk - 1] - G[j]) * kn[j][c];
            }
        }
        __syncthreads();
        // ---- A (strictly lower) and M (lower with diagonal): 16 dot products over the channels ----
        for (int p = warp; p < kBlk * (kBlk + 1) / 2 + kBlk * (kBlk - 1) / 2; p += NW) {
            // p < 10: M[i][j], j <= i; else A[i][j], j < i
            const bool isM = p < kBlk * (kBlk + 1) / 2;
            int q_ = isM ? p : p - kBlk * (kBlk + 1) / 2, i = 0;
            const int off = isM ? 0 : 1;
            while (q_ >= i + 1 - off) { q_ -= i + 1 - off; ++i; }
            const int j = q_;
            const float* x = isM ? qn[i] : kn[i];
            float part = 0.f;
            if (a.g_per_channel) {
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const int c = c0 + e;
                    part += x[c] * kn[j][c] * __expf(Gs[i][c] - Gs[j][c]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPT; ++e) part += x[c0 + e] * kn[j][c0 + e];
            }
            part = warp_sum(part);
            if (!a.g_per_channel) part *= __expf(Gs[i][0] - Gs[j][0]);
            if (lane == 0) {
                if (isM) Mm[i][j] = part;
                else Am[i][j] = bet[i] * part;
            }
        }
        __syncthreads();
        // ---- T = (I + A)^-1 (unit lower, forward substitution) and the U coefficients T diag(beta) ----
        if (tid == 0) {
            float T[kBlk][kBlk];
#pragma unroll
            for (int i = 0; i < kBlk; ++i)
#pragma unroll
                for (int j = 0; j < kBlk; ++j) T[i][j] = i == j ? 1.f : 0.f;
#pragma unroll
            for (int i = 1; i < kBlk; ++i)
#pragma unroll
                for (int j = 0; j < i; ++j) {
                    float acc = 0.f;
#pragma unroll
                    for (int m = j; m < i; ++m) acc += Am[i][m] * T[m][j];
                    T[i][j] = -acc;
                }
#pragma unroll
            for (int i = 0; i < kBlk; ++i)
#pragma unroll
                for (int j = 0; j < kBlk; ++j) Uc[i][j] = T[i][j] * bet[j];
        }
        __syncthreads();
        if (tid < D) {  // W_i = sum_j T[i][j] beta_j (e^G_j . k_j), in place per channel
            const int c = tid;
            float kg[kBlk];
#pragma unroll
            for (int j = 0; j < kBlk; ++j) kg[j] = Wm[j][c];
#pragma unroll
            for (int i = 0; i < kBlk; ++i) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j <= i; ++j) acc += Uc[i][j] * kg[j];
                Wm[i][c] = acc;
            }
        }
        __syncthreads();
        // ---- the unit's state rows: s_r . W_i and s_r . (e^G_i . q_i) for the block's tokens ----
        float dd[kBlk];
#pragma unroll
        for (int i = 0; i < kBlk; ++i) {
            float wv[EPT], qd[EPT];
#pragma unroll
            for (int e = 0; e < EPT; ++e) { wv[e] = Wm[i][c0 + e]; qd[e] = Qd[i][c0 + e]; }
            float x[32];
#pragma unroll
            for (int rr = 0; rr < kRowsPerWarp; ++rr) {
                float2 pk = make_float2(0.f, 0.f), pq = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < EPT; e += 2) {
                    const float2 sv = make_float2(s[rr][e], s[rr][e + 1]);
                    pk = __ffma2_rn(sv, make_float2(wv[e], wv[e + 1]), pk);
                    pq = __ffma2_rn(sv, make_float2(qd[e], qd[e + 1]), pq);
                }
                x[rr] = pk.x + pk.y;
                x[kRowsPerWarp + rr] = pq.x + pq.y;
            }
            dd[i] = transpose_reduce32(x, lane);  // lane < 16: s_r . W_i; lane >= 16: s_r . Qd_i (r = vrow)
        }
        // both halves of the warp get both products of row vrow, then V_new and y of that row
        float vn[kBlk], yv[kBlk];
#pragma unroll
        for (int i = 0; i < kBlk; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, dd[i], kRowsPerWarp);
            const float sw = lane < kRowsPerWarp ? dd[i] : other;   // s_r . W_i
            const float sq = lane < kRowsPerWarp ? other : dd[i];   // s_r . Qd_i
            float u = 0.f;
#pragma unroll
            for (int j = 0; j <= i; ++j) u += Uc[i][j] * vv[j][vrow];
            vn[i] = u - sw;
            float y = sq;
#pragma unroll
            for (int j = 0; j <= i; ++j) y += Mm[i][j] * vn[j];
            yv[i] = y;
        }
        // outputs, or for the gate each warp's sum of y^2 over its 16 rows (lanes < 16)
#pragma unroll
        for (int i = 0; i < kBlk; ++i) {
            const int t = t0 + i;
            const long vt = ((long)n * a.T + t) * a.H + h;
            if constexpr (GATE) {
                float sq = lane < kRowsPerWarp ? yv[i] * yv[i] : 0.f;
#pragma unroll
                for (int o = kRowsPerWarp / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
                if (lane == 0) part[i][warp] = sq;
            } else {
                if (t < a.T && (lane >> 4) == (i & 1)) store_out(a.out, vt * D + vrow, a.out_dtype, yv[i]);
            }
        }
        // ---- state update: s_r <- e^G_last . s_r + sum_j V_new[j][r] (e^(G_last - G_j) . k_j) ----
        {
            float gl[EPT], kd[kBlk][EPT];
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                gl[e] = gL[c0 + e];
#pragma unroll
                for (int j = 0; j < kBlk; ++j) kd[j][e] = Kd[j][c0 + e];
            }
#pragma unroll
            for (int rr = 0; rr < kRowsPerWarp; ++rr) {
                float vj[kBlk];
#pragma unroll
                for (int j = 0; j < kBlk; ++j) vj[j] = __shfl_sync(0xffffffffu, vn[j], rr);
#pragma unroll
                for (int e = 0; e < EPT; e += 2) {
                    float2 acc = __fmul2_rn(make_float2(gl[e], gl[e + 1]), make_float2(s[rr][e], s[rr][e + 1]));
#pragma unroll
                    for (int j = 0; j < kBlk; ++j)
                        acc = __ffma2_rn(make_float2(vj[j], vj[j]), make_float2(kd[j][e], kd[j][e + 1]), acc);
                    s[rr][e] = acc.x;
                    s[rr][e + 1] = acc.y;
                }
            }
        }
        if constexpr (GATE) {
            __syncthreads();  // every warp's partial sums are in
            if (lane < kRowsPerWarp) {
                const float w = a.w ? a.w[vrow] : 1.0f;
#pragma unroll
                for (int i = 0; i < kBlk; ++i) {
                    const int t = t0 + i;
                    if (t < a.T) {
                        float ss = 0.f;
#pragma unroll
                        for (int ww = 0; ww < NW; ++ww) ss += part[i][ww];
                        const long vt = ((long)n * a.T + t) * a.H + h;
                        const float z = zz[i][vrow];
                        store_out(a.out, vt * D + vrow, a.out_dtype,
                                  w * yv[i] * rsqrtf(ss / D + a.eps) * z * sigmoidf_(z));
                    }
                }
            }
        }
        __syncthreads();  // the block's shared rows are rewritten by the next block
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) StateVec<EPT>::store(S + (long)i * D, s[i]);

    if constexpr (CONV) {
        // final history: raw inputs of tokens T-3 .. T-1 (from the history when T < 3); every read
        // of the input history happened before the barrier that ended the first block
        if (a.conv.state_out && warp == 0) {
            float* so = a.conv.state_out + (long)slot * a.conv.dim * 3;
            float hq[3][EPT], hkk[3][EPT], hv[3][EPT];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int tau = a.T - 3 + j;
                if (tau >= 0) {
                    const long tk = (long)n * a.T + tau;
                    load_vec<EPT>(static_cast<const TIn*>(a.q) + (tk * a.Hk + hk) * D + c0, hq[j]);
                    load_vec<EPT>(static_cast<const TIn*>(a.k) + (tk * a.Hk + hk) * D + c0, hkk[j]);
                    load_vec<EPT>(static_cast<const TIn*>(a.v) + (tk * a.H + h) * D + c0, hv[j]);
                } else {
#pragma unroll
                    for (int e = 0; e < EPT; ++e) {
                        hq[j][e] = cs_in ? cs_in[(long)(cq + e) * 3 + 3 + tau] : 0.f;
                        hkk[j][e] = cs_in ? cs_in[(long)(ck + e) * 3 + 3 + tau] : 0.f;
                        hv[j][e] = cs_in ? cs_in[(long)(cv + e) * 3 + 3 + tau] : 0.f;
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < EPT; ++e)
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    if (h % grp == 0) {  // one writer per query/key head
                        so[(long)(cq + e) * 3 + j] = hq[j][e];
                        so[(long)(ck + e) * 3 + j] = hkk[j][e];
                    }
                    so[(long)(cv + e) * 3 + j] = hv[j][e];
                }
        }
    }
}

template <int D, typename TIn, bool GATE, bool CONV>
cudaError_t launch_variant(const DecodeArgs& a, cudaStream_t s, bool blocks) {
    const unsigned units = (unsigned)((long)a.N * a.H);
    if (blocks) decode_block_kernel<D, TIn, GATE, CONV><<<units, D * 2, 0, s>>>(a);
    else decode_kernel<D, TIn, GATE, CONV><<<units, D * 2, 0, s>>>(a);
    return cudaGetLastError();
}

// The block form when a unit's tokens fill its blocks to within one token, or there are many of
// them; otherwise token by token.  Measured (N = 256, H = 32, d = 128, bf16, gate; ms):
// T = 2: 0.222 vs 0.265 (blocks), 3: 0.292 vs 0.270, 4: 0.347 vs 0.272, 5: 0.404 vs 0.448,
// 8: 0.565 vs 0.467: a block costs about 0.19 ms here, a token about 0.06 ms.
// gdn_set_kernel_forms can force either form (for comparisons and tests).
template <int D, typename TIn>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    bool blocks = a.T >= 3 && (a.T % kBlk == 0 || a.T % kBlk == kBlk - 1 || a.T >= 10);
    const int form = decode_blocks_form();
    if (form != GDN_FORM_AUTO) blocks = form == GDN_FORM_ON && a.T >= 2;
    if (a.conv.w) {
        if (a.z) return launch_variant<D, TIn, true, true>(a, s, blocks);
        return launch_variant<D, TIn, false, true>(a, s, blocks);
    }
    if (a.z) return launch_variant<D, TIn, true, false>(a, s, blocks);
    return launch_variant<D, TIn, false, false>(a, s, blocks);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.d == 128) return a.qkv_dtype == GDN_BF16 ? launch_d<128, __nv_bfloat16>(a, s) : launch_d<128, float>(a, s);
    return a.qkv_dtype == GDN_BF16 ? launch_d<64, __nv_bfloat16>(a, s) : launch_d<64, float>(a, s);
}

}  // namespace gdn
