// decode.cu -- gated delta rule decode on kept fp32 states (gdn_recurrent_step and
// gdn_recurrent_multi_step: T tokens per sequence from a state pool, token by token in
// decode_kernel or, for several tokens or with the convolution, in decode_stream_kernel: blocks
// of four tokens in the chunked form, states staged through shared memory by bulk copies).
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
// HBM-bound: per (sequence, head) a call moves 2 * d_v * d_k * 4 bytes of state plus a few
// hundred bytes of q, k, v, y per token.  decode_kernel's layout: one CTA per (sequence, head); warp
// w owns 16 consecutive state rows; lane l holds d_k/32 consecutive columns of each row, so every
// row is one fully coalesced 128-bit (d_k = 128) or 64-bit (d_k = 64) access per lane.  All 16
// rows are loaded before any arithmetic (16 x 16 B in flight per lane).  The 32 dot products of
// a warp (16 rows x {k, q}) are reduced with a transposing butterfly: 31 shuffles leave dot
// product j on lane j, instead of 5 shuffles per dot product.
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

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

// ---- several tokens per unit, and the convolution: the streamed form ---------------------------
//
// "[LLM Algorithms-2] Gated DeltaNet" section 4 (the chunk form of the same recurrence) applied to
// a block of NB tokens of one unit, with S_0 the state before the block and, per key channel c,
// G_t[c] the block's cumulative log decay up to token t (one value for all channels when the decay
// is per head):
//     A[i][j] = beta_i sum_c k_i[c] k_j[c] e^(G_i - G_j)[c]   (j < i),   T = (I + A)^-1
//     W_i = sum_j T[i][j] beta_j (e^G_j . k_j),    U[i][r] = sum_j T[i][j] beta_j v_j[r]
//     V_new[i][r] = U[i][r] - s_r . W_i                       (s_r: state row r of S_0)
//     y_i[r] = s_r . (e^G_i . q_i) + sum_(j <= i) M[i][j] V_new[j][r],
//              M[i][j] = sum_c q_i[c] k_j[c] e^(G_i - G_j)[c]
//     s_r <- e^G_last . s_r + sum_j V_new[j][r] (e^(G_last - G_j) . k_j)
// which is the token-by-token update (prediction from the decayed state, write, read) regrouped,
// so a unit's tokens share one pass over its state: the 2 NB dot products of a state row are
// independent, and the update costs NB + 1 operations per element instead of 2 NB.  Every
// exponent is <= 0.  A block past the last token is padded with tokens that change nothing
// (k = q = v = 0, beta = 0, no decay), so any T works.  With NB = 1 the formulas are the
// single-token step itself (W = beta alpha k, U = beta v, M = q . k).
//
// Layout of the work.  Persistent CTAs (one per SM for d = 128, two for d = 64) take the (sequence,
// head) units with the grid as stride.  Each unit's state (64 KB at d = 128) is requested from HBM
// by bulk copies into a shared-memory stage kStages units ahead, so later units' reads are in
// flight while the current one computes.  The state warps (8 or 16 rows each, a row's columns over
// a half-warp) take the rows into registers, which frees the stage for the next request, run the
// unit's blocks and write the rows back to HBM from registers (for one-token blocks through an
// output buffer and bulk stores).  The block operands (W, U, e^G q, e^(G_last - G) k, e^G_last, M)
// depend on the inputs alone, so four preparing warps form them ahead of the state warps: block
// number b of the CTA (counted over its units) goes to preparing warp b mod 4, which writes it
// into a shared-memory slot of its own and so is never more than one use of that slot ahead.  Every wait is bounded; on a timeout the kernel records
// GDN_ERR_TIMEOUT, the state warps agree at the next unit to stop, and the requests still in
// flight are waited for (bounded) before the CTA exits.
constexpr int kBlk = 4;                      // tokens per block when a unit has several tokens
constexpr int kPrepWarps = 4;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on one mbarrier wait: 2 s

template <int D, int NB, bool GATE>
struct StreamShape {
    static constexpr int EPT = D / 32;
    // d = 128 without the gate: 16 state warps of 8 rows (more warps to hide the reductions'
    // latency); otherwise 16 rows a warp (the gate's per-block barrier over the state warps, and
    // d = 64 with two CTAs an SM, favour fewer warps)
    static constexpr bool kWide = D == 128 && !GATE;
    static constexpr int kRowsPerStateWarp = kWide ? 8 : 16;
    static constexpr int kStateWarps = D / kRowsPerStateWarp;
    static constexpr int kThreads = (kStateWarps + kPrepWarps) * 32;
    static constexpr int kCtasPerSm = D == 128 ? 1 : 2;
    // single-token blocks leave the state warps little arithmetic: their rows go back through an
    // output buffer by bulk stores, so the warps move on to the next unit at once
    static constexpr bool kOutBuf = NB == 1;
    // wide: launched at 96 registers a thread (640 threads); the state warpgroups give 8 back and
    // the preparing warpgroup takes 32 more (4 x 128 x 88 + 128 x 128 = 640 x 96)
    static constexpr bool kRegSplit = kWide;
    static constexpr int kRegsState = 88, kRegsPrep = 128;
    static_assert(!kRegSplit || (kStateWarps % 4 == 0 && 4 * 32 * (kStateWarps / 4) * kRegsState +
                                 4 * 32 * kRegsPrep == kThreads * 96), "register split");
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr uint32_t kState = D * D * 4;
    static constexpr uint32_t kCopy = kState < 16384 ? kState : 16384;  // bytes per bulk copy
    // a preparing warp's slot: W, e^G q, e^(G_last - G) k, U ([NB][D] each), e^G_last [D], the
    // gate input z [NB][D], M [NB][NB]
    static constexpr uint32_t kRows = NB * D * 4;
    static constexpr uint32_t oW = 0, oQd = kRows, oKd = 2 * kRows, oU = 3 * kRows, oGL = 4 * kRows;
    static constexpr uint32_t oZ = oGL + D * 4, oM = oZ + (GATE ? kRows : 0);
    static constexpr uint32_t kSlot = (oM + NB * NB * 4 + 15) / 16 * 16;
    // shared memory: state stages, slots, the gate's per-warp sums of squares [2][NB][warps], barriers
    static constexpr uint32_t oSlots = kStages * kState;
    static constexpr uint32_t oPart = oSlots + kPrepWarps * kSlot;
    static constexpr uint32_t oOut = oPart + 2 * NB * kStateWarps * 4;
    static constexpr uint32_t oBar = oOut + (kOutBuf ? kState : 0);
    static constexpr uint32_t kBytes = oBar + (kStages + 2 * kPrepWarps) * 8;
    static_assert(oOut % 16 == 0 && kState % kCopy == 0 && kBytes <= 232448, "layout");
};

template <int EPT>
__device__ __forceinline__ void lds_vec(const float* p, float* o) {
    if constexpr (EPT == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2*>(p);
        o[0] = t.x; o[1] = t.y;
    }
}
template <int EPT>
__device__ __forceinline__ void sts_vec(float* p, const float* o) {
    if constexpr (EPT == 4) *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
    else *reinterpret_cast<float2*>(p) = make_float2(o[0], o[1]);
}

// After this, lanes j and j + 16 hold the warp-wide sum of x[j] (16 values per lane in, 1 out).
// V values per lane in, 1 out: after this, lane l holds the sum over its half-warp (the 16 lanes
// with the same l >> 4) of x[l & (V - 1)].
template <int V>
__device__ __forceinline__ float transpose_reduce_half(float (&x)[V], int lane) {
#pragma unroll
    for (int width = V / 2; width >= 1; width >>= 1) {
        const bool upper = (lane & width) != 0;
#pragma unroll
        for (int j = 0; j < width; ++j) {
            float send = upper ? x[j] : x[j + width];
            float keep = upper ? x[j + width] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, width);
        }
    }
    float r = x[0];
#pragma unroll
    for (int o = V; o < 16; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}
// After this, lanes j and j + 16 hold the warp-wide sum of x[j].
__device__ __forceinline__ float transpose_reduce16(float (&x)[16], int lane) {
    const float h = transpose_reduce_half<16>(x, lane);
    return h + __shfl_xor_sync(0xffffffffu, h, 16);
}

// Pool slot of unit j's sequence, or -1 when the unit is skipped: a padding entry, or an index
// past the pool (recorded in `err` when given, so that one role reports it).
__device__ __forceinline__ int unit_slot(const DecodeArgs& a, int j, int* err) {
    const int n = j / a.H;
    const int s = a.idx ? a.idx[n] : n;
    if (s >= a.num_slots) {
        if (err) record_error(err, GDN_ERR_ARG);
        return -1;
    }
    return s;
}
// The first unit at or after j, in steps of the grid, that is not skipped; `units` when none is left.
__device__ __forceinline__ int next_unit(const DecodeArgs& a, int j, int units, int* slot, int* err) {
    for (; j < units; j += gridDim.x)
        if ((*slot = unit_slot(a, j, err)) >= 0) return j;
    return units;
}

// Forms block t0 .. t0 + NB - 1 of unit (n, h) in slot `sl` (one warp; lane holds key and value
// channels c0 .. c0 + EPT - 1).  With the convolution, the block at t0 = 0 also writes the unit's
// final history: only that block reads the input history (NB >= 3, or T = 1), and the lane that
// reads a channel's history is the one that writes it, after its reads, so the history may be
// updated in place.
template <int D, typename TIn, bool GATE, bool CONV, int NB>
__device__ __forceinline__ void prep_block(const DecodeArgs& a, uint8_t* sl, int n, int h, int slot, int t0,
                                           int lane) {
    using L = StreamShape<D, NB, GATE>;
    constexpr int EPT = L::EPT;
    const int grp = a.H / a.Hk, hk = h / grp, c0 = lane * EPT;
    const int cq = hk * D + c0, ck = a.Hk * D + cq, cv = 2 * a.Hk * D + h * D + c0;  // conv channels
    const float* cs_in = CONV && a.conv.state_in ? a.conv.state_in + (long)slot * a.conv.dim * 3 : nullptr;
    float qv[NB][EPT], kv[NB][EPT], vx[NB][EPT], G[NB][EPT], bt[NB];
    if constexpr (CONV) {
        // raw inputs of tokens t0 - 3 .. t0 + NB - 1: this call's, the history before it, zero after it
        float rq[NB + 3][EPT], rk[NB + 3][EPT], rv[NB + 3][EPT];
#pragma unroll
        for (int m = 0; m < NB + 3; ++m) {
            const int tau = t0 - 3 + m;
            if (tau >= 0 && tau < a.T) {
                const long tk = (long)n * a.T + tau;
                load_vec<EPT>(static_cast<const TIn*>(a.q) + (tk * a.Hk + hk) * D + c0, rq[m]);
                load_vec<EPT>(static_cast<const TIn*>(a.k) + (tk * a.Hk + hk) * D + c0, rk[m]);
                load_vec<EPT>(static_cast<const TIn*>(a.v) + (tk * a.H + h) * D + c0, rv[m]);
            } else {
                const bool hist = tau < 0 && cs_in;
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    rq[m][e] = hist ? cs_in[(long)(cq + e) * 3 + 3 + tau] : 0.f;
                    rk[m][e] = hist ? cs_in[(long)(ck + e) * 3 + 3 + tau] : 0.f;
                    rv[m][e] = hist ? cs_in[(long)(cv + e) * 3 + 3 + tau] : 0.f;
                }
            }
        }
        const float4* w4 = reinterpret_cast<const float4*>(a.conv.w);
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            const float4 wq = __ldg(w4 + cq + e), wk = __ldg(w4 + ck + e), wv = __ldg(w4 + cv + e);
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                const bool live = t0 + i < a.T;
                qv[i][e] = live ? round_to<TIn>(conv4_silu(wq, rq[i][e], rq[i + 1][e], rq[i + 2][e], rq[i + 3][e])) : 0.f;
                kv[i][e] = live ? round_to<TIn>(conv4_silu(wk, rk[i][e], rk[i + 1][e], rk[i + 2][e], rk[i + 3][e])) : 0.f;
                vx[i][e] = live ? round_to<TIn>(conv4_silu(wv, rv[i][e], rv[i + 1][e], rv[i + 2][e], rv[i + 3][e])) : 0.f;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int t = t0 + i;
            if (t < a.T) {
                const long tok = (long)n * a.T + t;
                load_vec<EPT>(static_cast<const TIn*>(a.q) + (tok * a.Hk + hk) * D + c0, qv[i]);
                load_vec<EPT>(static_cast<const TIn*>(a.k) + (tok * a.Hk + hk) * D + c0, kv[i]);
                load_vec<EPT>(static_cast<const TIn*>(a.v) + (tok * a.H + h) * D + c0, vx[i]);
            } else {
#pragma unroll
                for (int e = 0; e < EPT; ++e) qv[i][e] = kv[i][e] = vx[i][e] = 0.f;
            }
        }
    }
    // decay, beta, gate input; normalised k, scaled normalised q
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        const int t = t0 + i;
        const long vt = ((long)n * a.T + t) * a.H + h;
        if (t < a.T) {
            if (a.g_per_channel) {
                load_vec<EPT>(a.g + vt * D + c0, G[i]);
            } else {
                const float g0 = a.g[vt];
#pragma unroll
                for (int e = 0; e < EPT; ++e) G[i][e] = g0;
            }
            bt[i] = a.beta[vt];
        } else {
#pragma unroll
            for (int e = 0; e < EPT; ++e) G[i][e] = 0.f;
            bt[i] = 0.f;
        }
        if constexpr (GATE) {
            float zv[EPT];
            if (t < a.T) {
                load_vec<EPT>(a.z + vt * D + c0, zv);
            } else {
#pragma unroll
                for (int e = 0; e < EPT; ++e) zv[e] = 0.f;
            }
            sts_vec<EPT>(reinterpret_cast<float*>(sl + L::oZ) + i * D + c0, zv);
        }
        float ssq = 0.f, ssk = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { ssq += qv[i][e] * qv[i][e]; ssk += kv[i][e] * kv[i][e]; }
        ssq = warp_sum(ssq);
        ssk = warp_sum(ssk);
        const float qf = a.use_l2 ? a.scale * rsqrtf(ssq + kL2Eps) : a.scale;
        const float kf = a.use_l2 ? rsqrtf(ssk + kL2Eps) : 1.0f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) { qv[i][e] *= qf; kv[i][e] *= kf; }
    }
    // cumulative log decay over the block
#pragma unroll
    for (int i = 1; i < NB; ++i)
#pragma unroll
        for (int e = 0; e < EPT; ++e) G[i][e] += G[i - 1][e];
    // P[i][j] = q_i . k_j e^(G_i - G_j) (j <= i: M[i][j]) and k_j . k_i e^(G_j - G_i) (j > i:
    // A[j][i] / beta_j), over the channels; every exponent is <= 0
    float P[NB == 1 ? 1 : 16];
    static_assert(NB == 1 || NB == 4, "blocks of one or four tokens");
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                if (j <= i) acc += qv[i][e] * kv[j][e] * __expf(G[i][e] - G[j][e]);
                else acc += kv[j][e] * kv[i][e] * __expf(G[j][e] - G[i][e]);
            }
            P[i * NB + j] = acc;
        }
    float* Ms = reinterpret_cast<float*>(sl + L::oM);
    float Am[NB][NB];  // A[i][m], m < i, on every lane
    if constexpr (NB == 1) {
        const float m00 = warp_sum(P[0]);
        if (lane == 0) Ms[0] = m00;
    } else {
        const float red = transpose_reduce16(P, lane);  // lane l: P[l & 15]
        if (lane < NB * NB) Ms[lane] = (lane % NB <= lane / NB) ? red : 0.f;
#pragma unroll
        for (int i = 1; i < NB; ++i)
#pragma unroll
            for (int m = 0; m < i; ++m) Am[i][m] = bt[i] * __shfl_sync(0xffffffffu, red, m * NB + i);
    }
    // T = (I + A)^-1 (unit lower, forward substitution), then the coefficients T diag(beta)
    float Tm[NB][NB];
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
        for (int j = 0; j < NB; ++j) Tm[i][j] = i == j ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < NB; ++i)
#pragma unroll
        for (int j = 0; j < i; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int m = j; m < i; ++m) acc += Am[i][m] * Tm[m][j];
            Tm[i][j] = -acc;
        }
    // W_i, U_i, e^G_i q_i, e^(G_last - G_i) k_i, e^G_last
    float* Ws = reinterpret_cast<float*>(sl + L::oW);
    float* Qs = reinterpret_cast<float*>(sl + L::oQd);
    float* Ks = reinterpret_cast<float*>(sl + L::oKd);
    float* Us = reinterpret_cast<float*>(sl + L::oU);
    float eG[NB][EPT];
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
        for (int e = 0; e < EPT; ++e) eG[i][e] = __expf(G[i][e]);
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        float wr[EPT], ur[EPT], qd[EPT], kd[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            float aw = 0.f, au = 0.f;
#pragma unroll
            for (int j = 0; j <= i; ++j) {
                const float c = Tm[i][j] * bt[j];
                aw += c * (eG[j][e] * kv[j][e]);
                au += c * vx[j][e];
            }
            wr[e] = aw;
            ur[e] = au;
            qd[e] = eG[i][e] * qv[i][e];
            kd[e] = __expf(G[NB - 1][e] - G[i][e]) * kv[i][e];
        }
        sts_vec<EPT>(Ws + i * D + c0, wr);
        sts_vec<EPT>(Us + i * D + c0, ur);
        sts_vec<EPT>(Qs + i * D + c0, qd);
        sts_vec<EPT>(Ks + i * D + c0, kd);
    }
    sts_vec<EPT>(reinterpret_cast<float*>(sl + L::oGL) + c0, eG[NB - 1]);

    if constexpr (CONV) {
        // final history: raw inputs of tokens T-3 .. T-1 (from the history when T < 3); all reads first
        if (t0 == 0 && a.conv.state_out) {
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

template <int D, typename TIn, bool GATE, bool CONV, int NB>
__global__ void __launch_bounds__(StreamShape<D, NB, GATE>::kThreads, StreamShape<D, NB, GATE>::kCtasPerSm)
    decode_stream_kernel(DecodeArgs a) {
    using L = StreamShape<D, NB, GATE>;
    constexpr int WS = L::kStateWarps;
    extern __shared__ __align__(128) uint8_t sm[];
    uint64_t* sfull = reinterpret_cast<uint64_t*>(sm + L::oBar);  // [kStages] state copies landed
    uint64_t* pfull = sfull + L::kStages;                          // [4] a preparing warp's slot written
    uint64_t* pempty = pfull + kPrepWarps;                         // [4] the slot read by every state warp
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int units = a.N * a.H, nb = (a.T + NB - 1) / NB, grid = gridDim.x;
    if (tid == 0) {
        for (int s = 0; s < L::kStages; ++s) ptx::mbar_init(&sfull[s], 1);
        for (int p = 0; p < kPrepWarps; ++p) {
            ptx::mbar_init(&pfull[p], 32);
            ptx::mbar_init(&pempty[p], WS);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp >= WS) {
        // ---- preparing warps: block b of the CTA's sequence of blocks by warp b mod 4 ----
        if constexpr (L::kRegSplit) ptx::reg_alloc<L::kRegsPrep>();
        const int pw = warp - WS;
        int b = 0;
        for (int j = blockIdx.x, slot; (j = next_unit(a, j, units, &slot, nullptr)) < units; j += grid) {
            for (int blk = 0; blk < nb; ++blk, ++b) {
                if (b % kPrepWarps != pw) continue;
                const int use = b / kPrepWarps;
                if (use > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(&pempty[pw], (use - 1) & 1, kWaitNs))) {
                    if (lane == 0) record_error(a.err, GDN_ERR_TIMEOUT);
                    return;
                }
                prep_block<D, TIn, GATE, CONV, NB>(a, sm + L::oSlots + pw * L::kSlot, j / a.H, j % a.H, slot, blk * NB,
                                                   lane);
                ptx::mbar_arrive(&pfull[pw]);  // every lane: its slot writes are released
            }
        }
        return;
    }

    // ---- state warps ----
    // Warp w owns rows r0 .. r0 + RW - 1; lane l holds rows r0 + RPH (l >> 4) + m (m < RPH), and of
    // each row the column chunks 64 k + 4 (l & 15) .. + 3 (k < D / 64), so a row's dot product is
    // spread over the 16 lanes of a half-warp and every shared or global access of a half-warp to
    // one row is 256 contiguous bytes.  After the reductions, the lanes of a half-warp with the
    // same l mod RPH hold one row: bit RPH tells s_r . W from s_r . (e^G q), the bits above it
    // number the copies, which share that row's output stores.
    if constexpr (L::kRegSplit) ptx::reg_dealloc<L::kRegsState>();
    constexpr int RW = L::kRowsPerStateWarp, RPH = RW / 2, V = 2 * RPH;
    constexpr int CH = D / 64, CPL = 4 * CH;  // float4 chunks and columns per lane and row
    constexpr int kGroups = 16 / RPH;         // lanes of a half-warp that share a row
    const int r0 = warp * RW, hf = lane >> 4, cs = lane & 15;
    const int rl = RPH * hf + (lane & (RPH - 1));  // the row whose V_new and y this lane forms
    const bool wside = (lane & RPH) == 0;
    const int grpid = cs / RPH;                    // 0 .. kGroups - 1
    float* part = reinterpret_cast<float*>(sm + L::oPart);
    auto ld_cols = [&](const float* row, float* o) {  // this lane's columns of a row in shared memory
#pragma unroll
        for (int k = 0; k < CH; ++k) lds_vec<4>(row + 64 * k + 4 * cs, o + 4 * k);
    };
    // thread 0 requests the states: the k-th request goes to stage k mod kStages
    int pj = blockIdx.x, issued = 0;
    auto request = [&](int stage) {
        int ps;
        pj = next_unit(a, pj, units, &ps, a.err);
        if (pj >= units) return;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.state + ((long)ps * a.H + pj % a.H) * D * D);
        uint8_t* dst = sm + stage * L::kState;
        ptx::mbar_arrive_expect_tx(&sfull[stage], L::kState);
#pragma unroll
        for (uint32_t o = 0; o < L::kState; o += L::kCopy) ptx::bulk_load(dst + o, src + o, L::kCopy, &sfull[stage]);
        pj += grid;
        ++issued;
    };
    if (tid == 0)
        for (int st = 0; st < L::kStages; ++st) request(st);

    int ui = 0, b = 0;
    bool bad = false;
    float s[RPH][CPL];
    for (int j = blockIdx.x, slot; (j = next_unit(a, j, units, &slot, nullptr)) < units; j += grid, ++ui) {
        const int n = j / a.H, h = j % a.H, st = ui % L::kStages;
        const bool landed = !bad && ptx::mbar_wait(&sfull[st], (ui / L::kStages) & 1, kWaitNs);
        if (landed) {
            const float* src = reinterpret_cast<const float*>(sm + st * L::kState) + (r0 + RPH * hf) * D;
#pragma unroll
            for (int m = 0; m < RPH; ++m) ld_cols(src + m * D, s[m]);
        }
        // every state warp has its rows (the stage is free), or all stop together
        if (ptx::bar_sync_or(1, WS * 32, !landed)) {
            bad = true;
            break;
        }
        // four-token blocks: the next state is requested at once.  One-token blocks have little
        // arithmetic between the copy-out and the write-back, and a request issued at once competed
        // with that write-back and the convolution history's traffic (0.212 against 0.190 ms for the
        // convolution step at N = 256, H = 32): they request after the block.
        if constexpr (NB != 1) {
            if (tid == 0) request(st);
        }

        for (int blk = 0; blk < nb; ++blk, ++b) {
            const int w = b % kPrepWarps, t0 = blk * NB;
            const bool ready = !bad && __all_sync(0xffffffffu, ptx::mbar_wait(&pfull[w], (b / kPrepWarps) & 1, kWaitNs));
            bad = !ready;
            const uint8_t* sl = sm + L::oSlots + w * L::kSlot;
            const float* Ms = reinterpret_cast<const float*>(sl + L::oM);
            float yv[NB];
            if (ready) {
                // s_r . W_i and s_r . (e^G_i q_i) for the block's tokens
                const float* Ws = reinterpret_cast<const float*>(sl + L::oW);
                const float* Qs = reinterpret_cast<const float*>(sl + L::oQd);
                const float* Us = reinterpret_cast<const float*>(sl + L::oU);
                float dd[NB];
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                    float wv[CPL], qd[CPL];
                    ld_cols(Ws + i * D, wv);
                    ld_cols(Qs + i * D, qd);
                    float x[V];
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        float2 pk = make_float2(0.f, 0.f), pq = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < CPL; e += 2) {
                            const float2 sv = make_float2(s[m][e], s[m][e + 1]);
                            pk = __ffma2_rn(sv, make_float2(wv[e], wv[e + 1]), pk);
                            pq = __ffma2_rn(sv, make_float2(qd[e], qd[e + 1]), pq);
                        }
                        x[m] = pk.x + pk.y;
                        x[RPH + m] = pq.x + pq.y;
                    }
                    dd[i] = transpose_reduce_half<V>(x, lane);
                }
                // both sides of a row get both of its products, then V_new and y of that row
                float vn[NB];
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                    const float other = __shfl_xor_sync(0xffffffffu, dd[i], RPH);
                    const float sw = wside ? dd[i] : other;
                    const float sq = wside ? other : dd[i];
                    vn[i] = Us[i * D + r0 + rl] - sw;
                    float y = sq;
#pragma unroll
                    for (int j2 = 0; j2 <= i; ++j2) y += Ms[i * NB + j2] * vn[j2];
                    yv[i] = y;
                }
                // s_r <- e^G_last . s_r + sum_j V_new[j][r] (e^(G_last - G_j) . k_j), a column pair at a time
                const float* Ks = reinterpret_cast<const float*>(sl + L::oKd);
                const float* GLs = reinterpret_cast<const float*>(sl + L::oGL);
                float vj[RPH][NB];
#pragma unroll
                for (int m = 0; m < RPH; ++m)
#pragma unroll
                    for (int j2 = 0; j2 < NB; ++j2) vj[m][j2] = __shfl_sync(0xffffffffu, vn[j2], (lane & 16) | m);
#pragma unroll
                for (int e = 0; e < CPL; e += 2) {
                    const int col = 64 * (e / 4) + 4 * cs + (e & 3);
                    const float2 g2 = *reinterpret_cast<const float2*>(GLs + col);
                    float2 k2[NB];
#pragma unroll
                    for (int j2 = 0; j2 < NB; ++j2) k2[j2] = *reinterpret_cast<const float2*>(Ks + j2 * D + col);
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        float2 acc = __fmul2_rn(g2, make_float2(s[m][e], s[m][e + 1]));
#pragma unroll
                        for (int j2 = 0; j2 < NB; ++j2) acc = __ffma2_rn(make_float2(vj[m][j2], vj[m][j2]), k2[j2], acc);
                        s[m][e] = acc.x;
                        s[m][e + 1] = acc.y;
                    }
                }
                if constexpr (!GATE) {  // the kGroups copies of a row share its tokens' stores
#pragma unroll
                    for (int i = 0; i < NB; ++i) {
                        const int t = t0 + i;
                        if (t < a.T && grpid == i % kGroups)
                            store_out(a.out, (((long)n * a.T + t) * a.H + h) * D + r0 + rl, a.out_dtype, yv[i]);
                    }
                }
            }
            if constexpr (GATE) {
                // RMS over the d_v rows of each token: per-warp sums of squares, one barrier per block
                // (two buffers, so a warp that runs ahead never overwrites sums still being read)
                float* pp = part + (b & 1) * NB * WS;
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                    float sq = ready && grpid == 0 ? yv[i] * yv[i] : 0.f;
                    sq = warp_sum(sq);
                    if (lane == 0) pp[i * WS + warp] = sq;
                }
                ptx::bar_sync(2, WS * 32);
                if (ready) {
                    const float* Zs = reinterpret_cast<const float*>(sl + L::oZ);
                    const int r = r0 + rl;
                    const float wr = a.w ? a.w[r] : 1.0f;
#pragma unroll
                    for (int i = 0; i < NB; ++i) {
                        const int t = t0 + i;
                        if (t < a.T && grpid == i % kGroups) {
                            float ss = 0.f;
#pragma unroll
                            for (int ww = 0; ww < WS; ++ww) ss += pp[i * WS + ww];
                            const float z = Zs[i * D + r];
                            store_out(a.out, (((long)n * a.T + t) * a.H + h) * D + r, a.out_dtype,
                                      wr * yv[i] * rsqrtf(ss / D + a.eps) * z * sigmoidf_(z));
                        }
                    }
                }
            }
            if (ready) {
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&pempty[w]);
            }
        }
        if constexpr (NB == 1) {
            if (tid == 0) request(st);
        }
        if constexpr (L::kOutBuf) {
            // the rows go through the output buffer and leave by bulk stores
            if (tid == 0) ptx::bulk_wait_read();  // the previous unit's rows have left the buffer
            if (ptx::bar_sync_or(3, WS * 32, bad)) {
                bad = true;
                continue;
            }
            float* ob = reinterpret_cast<float*>(sm + L::oOut) + (r0 + RPH * hf) * D + 4 * cs;
#pragma unroll
            for (int m = 0; m < RPH; ++m)
#pragma unroll
                for (int k = 0; k < CH; ++k) sts_vec<4>(ob + m * D + 64 * k, s[m] + 4 * k);
            ptx::fence_async_smem();
            ptx::bar_sync(3, WS * 32);
            if (tid == 0) {
                uint8_t* S = reinterpret_cast<uint8_t*>(a.state + ((long)slot * a.H + h) * D * D);
#pragma unroll
                for (uint32_t o = 0; o < L::kState; o += L::kCopy) ptx::bulk_store(S + o, sm + L::oOut + o, L::kCopy);
                ptx::bulk_commit();
            }
        } else if (!bad) {
            float* S = a.state + ((long)slot * a.H + h) * D * D + (long)(r0 + RPH * hf) * D + 4 * cs;
#pragma unroll
            for (int m = 0; m < RPH; ++m)
#pragma unroll
                for (int k = 0; k < CH; ++k) StateVec<4>::store(S + (long)m * D + 64 * k, s[m] + 4 * k);
        }
    }
    if (bad && lane == 0) record_error(a.err, GDN_ERR_TIMEOUT);
    // requests not consumed (only after a timeout) are waited for before the CTA exits
    if (tid == 0) {
        for (int k = ui; k < issued; ++k) ptx::mbar_wait(&sfull[k % L::kStages], (k / L::kStages) & 1, kWaitNs);
        if constexpr (L::kOutBuf) ptx::bulk_wait_all();  // the last rows are written before the CTA exits
    }
}

template <int D, typename TIn, bool GATE, bool CONV, int NB>
cudaError_t launch_stream(const DecodeArgs& a, cudaStream_t s) {
    using L = StreamShape<D, NB, GATE>;
    auto* fn = decode_stream_kernel<D, TIn, GATE, CONV, NB>;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes)) != cudaSuccess)
        return e;
    const long units = (long)a.N * a.H, cap = (long)sms * L::kCtasPerSm;
    fn<<<(unsigned)(units < cap ? units : cap), L::kThreads, L::kBytes, s>>>(a);
    return cudaGetLastError();
}

template <int D, typename TIn, bool GATE, bool CONV>
cudaError_t launch_variant(const DecodeArgs& a, cudaStream_t s, bool stream) {
    if (!stream) {
        decode_kernel<D, TIn, GATE, CONV><<<(unsigned)((long)a.N * a.H), D * 2, 0, s>>>(a);
        return cudaGetLastError();
    }
    if (a.T == 1) return launch_stream<D, TIn, GATE, CONV, 1>(a, s);
    return launch_stream<D, TIn, GATE, CONV, kBlk>(a, s);
}

// The streamed form for several tokens per unit and for the convolution; one token without the
// convolution goes token by token (decode_kernel: load, one update, store, already at the copy
// rate).  gdn_set_kernel_forms can force either form (for comparisons and tests).
template <int D, typename TIn>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    bool stream = a.T >= 2 || a.conv.w;
    const int form = decode_blocks_form();
    if (form != GDN_FORM_AUTO) stream = form == GDN_FORM_ON;
    if (a.conv.w) {
        if (a.z) return launch_variant<D, TIn, true, true>(a, s, stream);
        return launch_variant<D, TIn, false, true>(a, s, stream);
    }
    if (a.z) return launch_variant<D, TIn, true, false>(a, s, stream);
    return launch_variant<D, TIn, false, false>(a, s, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.d == 128) return a.qkv_dtype == GDN_BF16 ? launch_d<128, __nv_bfloat16>(a, s) : launch_d<128, float>(a, s);
    return a.qkv_dtype == GDN_BF16 ? launch_d<64, __nv_bfloat16>(a, s) : launch_d<64, float>(a, s);
}

}  // namespace gdn
