// prefill_tc.cu -- chunked prefill on the tcgen05 tensor cores (gdn_chunk_fwd, bf16 q/k/v, d = 128).
//
// Algorithm: "5. 线性注意力", "Delta Rule 的 Chunk 实现" (chunks of C = 64 tokens).  Notation per
// chunk of one (sequence, head): K, Q, V the raw 64 x 128 tiles, kinv_i = 1/||k_i||,
// qs_i = scale/||q_i|| (L2 normalisation folded into per-row factors instead of rewriting the
// tiles), gc the inclusive cumulative sum of g, D_ij = exp(gc_i - gc_j) for i >= j.
//   A_ij   = beta_i D_ij kinv_i kinv_j (k_i . k_j)        j < i     (from K K^T)
//   T      = (I + A)^-1                                             (fp32, CUDA cores)
//   W      = T diag(beta e^gc kinv) K     (= T diag(beta e^gc) K_normalised)
//   U      = T diag(beta) V
//   Aqk_ij = D_ij qs_i kinv_j (q_i . k_j)                  j <= i    (from Q K^T)
//   V_new  = U - W S^T
//   O      = diag(e^gc qs) Q S^T + Aqk V_new
//   S'     = e^{gc_last} S + V_new^T diag(e^{gc_last - gc} kinv) K
//
// Three launches on the caller's stream:
//   chunk_map_kernel    numbers the chunks of all sequences (varlen) in the workspace.
//   chunk_prep_kernel   one CTA per (chunk, head), all in parallel: TMA loads of K, Q, V; one MMA
//                       [K;Q][K;Q]^T (M=128, N=128, K=128); the triangular solve on the CUDA
//                       cores; two MMAs W^T = K^T T'^T and U^T = V^T T''^T (MN-major A from the
//                       same K / V tiles); W, U^T, Aqk (bf16) and per-token factors to workspace.
//   chunk_state_kernel  one CTA per (sequence, head), walking the chunks in order, warp-specialised:
//                       warp 0 issues TMA loads of the next chunk's operands (two-stage ring),
//                       warp 1 issues the MMAs (warps 0-3 run with few registers), warps 4-7 run
//                       the state epilogue (the serial chain: V_new, then S), warps 8-11 the
//                       output epilogue (O and the fused RMSNorm * SiLU gate).  The state S is fp32 in TMEM (lanes = rows d_v,
//                       columns = d_k) and is mirrored as a bf16 operand tile in shared memory.
//   TMEM per state CTA: S [0,128), two buffers of S [W;Q]^T [128,384), two of A1 Aqk^T [384,512).
//
// Every mbarrier wait is bounded; on a timeout the kernel records GDN_ERR_TIMEOUT and its roles
// stop issuing work, wait (bounded) for what they issued, free TMEM and return.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr uint64_t kPolls = 2000000000ull;  // bound on any single mbarrier wait: 2 s of wall time

// ---- workspace layout --------------------------------------------------------------------------

struct WsLayout {
    long nch;          // chunk-head slots = max_chunks * H
    size_t off_map, off_first, off_count, off_W, off_Ut, off_Aqk, off_scal, total;
};

__host__ __device__ inline long max_chunks(int num_seqs, int total_T) { return (long)total_T / kC + num_seqs; }

inline WsLayout ws_layout(int num_seqs, int total_T, int H) {
    WsLayout w{};
    const long mc = max_chunks(num_seqs, total_T);
    w.nch = mc * H;
    auto al = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    size_t o = 0;
    w.off_map = o;   o = al(o + sizeof(int32_t) * mc);               // chunk -> sequence
    w.off_first = o; o = al(o + sizeof(int32_t) * (num_seqs + 1));   // first chunk of each sequence
    w.off_count = o; o = al(o + sizeof(int32_t) * 4);                 // number of chunks
    w.off_W = o;     o = al(o + sizeof(__nv_bfloat16) * w.nch * kC * kD);
    w.off_Ut = o;    o = al(o + sizeof(__nv_bfloat16) * w.nch * kD * kC);
    w.off_Aqk = o;   o = al(o + sizeof(__nv_bfloat16) * w.nch * kC * kC);
    w.off_scal = o;  o = al(o + sizeof(float) * w.nch * 4 * kC);
    w.total = o;
    return w;
}

struct TcArgs {
    const int32_t* cu;   // may be null: fixed length
    int num_seqs, total_T, H;
    const float* g;
    const float* beta;
    float scale;
    int use_l2;
    int32_t* chunk_seq;
    int32_t* chunk_first;
    int32_t* n_chunks;
    __nv_bfloat16* W;
    __nv_bfloat16* Ut;
    __nv_bfloat16* Aqk;
    float* scal;
    const float* initial_state;
    float* final_state;
    const float* z;
    const float* w;
    float eps;
    void* out;
    gdn_dtype out_dtype;
    int* err;
};

__device__ __forceinline__ bool seq_bounds(const TcArgs& a, int n, long& bos, long& eos) {
    if (a.cu) {
        bos = a.cu[n];
        eos = a.cu[n + 1];
        return !(bos < 0 || eos < bos || eos > a.total_T);
    }
    const long T = a.total_T / a.num_seqs;
    bos = (long)n * T;
    eos = bos + T;
    return true;
}

// ---- 1. chunk map --------------------------------------------------------------------------------

__global__ void __launch_bounds__(1024) chunk_map_kernel(TcArgs a) {
    __shared__ int32_t part[1024];
    const int tid = threadIdx.x;
    // per-thread contiguous block of sequences
    const int per = (a.num_seqs + 1023) / 1024;
    const int s0 = tid * per, s1 = min(a.num_seqs, s0 + per);
    int32_t cnt = 0;
    for (int n = s0; n < s1; ++n) {
        long bos, eos;
        if (seq_bounds(a, n, bos, eos)) cnt += (int32_t)((eos - bos + kC - 1) / kC);
        else record_error(a.err, GDN_ERR_CU_SEQLENS);
    }
    part[tid] = cnt;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan
        int32_t t = tid >= o ? part[tid - o] : 0;
        __syncthreads();
        part[tid] += t;
        __syncthreads();
    }
    int32_t base = part[tid] - cnt;
    for (int n = s0; n < s1; ++n) {
        long bos, eos;
        int32_t c = seq_bounds(a, n, bos, eos) ? (int32_t)((eos - bos + kC - 1) / kC) : 0;
        a.chunk_first[n] = base;
        for (int32_t j = 0; j < c; ++j) a.chunk_seq[base + j] = n;
        base += c;
    }
    if (tid == 1023) {
        a.chunk_first[a.num_seqs] = part[1023];
        a.n_chunks[0] = part[1023];
    }
}

// ---- shared helpers --------------------------------------------------------------------------------

// logistic function for the output gate (its result is rounded to the output type right after)
__device__ __forceinline__ float fast_sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

// write 8 consecutive bf16 (one 16-byte chunk) of row `row` at column 8*chunk of a SW128 tile
__device__ __forceinline__ void st_sw128_chunk(uint8_t* tile, int row, int chunk, const float* v) {
    uint4 p;
    p.x = pack_bf16x2(v[0], v[1]);
    p.y = pack_bf16x2(v[2], v[3]);
    p.z = pack_bf16x2(v[4], v[5]);
    p.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, chunk * 8)) = p;
}

__device__ __forceinline__ void ld_sw128_chunk(const uint8_t* tile, int row, int chunk, float* v) {
    uint4 p = *reinterpret_cast<const uint4*>(tile + sw128_offset(row, chunk * 8));
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
        float2 f = __bfloat1622float2(t);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

// ---- 2. chunk preparation (parallel) ------------------------------------------------------------

namespace prep {
constexpr int kThreads = 128;
constexpr int LD = kC + 1;  // padded fp32 64x64 tiles
constexpr uint32_t oKQ = 0;          // 2 atom columns x (K rows 0-63, Q rows 64-127) = 32 KB
constexpr uint32_t oV = 32768;       // 2 atom columns x 64 rows = 16 KB
constexpr uint32_t oTP = 49152;      // T' (bf16 SW128 64x64) 8 KB
constexpr uint32_t oTPP = 57344;     // T'' 8 KB
constexpr uint32_t oAf = 65536;      // A (fp32 64 x 65); later the W staging tile (bf16 64x128)
constexpr uint32_t oTf = oAf + 4 * kC * LD;       // T (fp32 64 x 65)
constexpr uint32_t oSc = oTf + 4 * kC * LD;       // gc, beta, kinv, qs (fp32 x 64 each)
constexpr uint32_t oBar = oSc + 4 * 4 * kC;       // 2 mbarriers + TMEM base
constexpr uint32_t kBytes = oBar + 64;
constexpr uint32_t kSmem = kBytes + 1024;          // + alignment slack
constexpr uint32_t kTmemCols = 256;
}  // namespace prep

// Blocked inverse of the unit lower-triangular 64x64 matrix I + A (A strictly lower, fp32 in Af with
// row stride LD) into Tf.  Diagonal 16x16 blocks by forward substitution (one warp per block, one
// lane per column), then block rows 1..3 by T_bj = -T_bb sum_{k=j}^{b-1} A_bk T_kj.
__device__ void unit_lower_inverse(const float* Af, float* Tf, float* X, int tid) {
    constexpr int LD = prep::LD;
    const int warp = tid >> 5, lane = tid & 31;
    {   // diagonal blocks
        const int b0 = warp * 16;
        if (lane < 16) {
            const int jj = lane;
            float t[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < ii; ++m)
                    if (m >= jj) acc += Af[(b0 + ii) * LD + b0 + m] * t[m];
                t[ii] = ii < jj ? 0.f : (ii == jj ? 1.f : -acc);
            }
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) Tf[(b0 + ii) * LD + b0 + jj] = t[ii];
        }
        // zero the strictly upper blocks of this block row
        for (int e = lane; e < 16 * 64; e += 32) {
            const int ii = e / 64, j = e % 64;
            if (j >= b0 + 16) Tf[(b0 + ii) * LD + j] = 0.f;
        }
    }
    bar_sync(2, prep::kThreads);
    for (int b = 1; b < 4; ++b) {
        const int nel = b * 256;  // elements of block row b left of the diagonal
        // X_bj = sum_{k=j}^{b-1} A_bk T_kj   (16 x 16 each), stored in X[16][b*16]
        for (int e = tid; e < nel; e += prep::kThreads) {
            const int ii = e / (b * 16), col = e % (b * 16);  // col in [0, 16b)
            const int j = col / 16;
            float acc = 0.f;
            for (int m = j * 16; m < b * 16; ++m) acc += Af[(b * 16 + ii) * LD + m] * Tf[m * LD + col];
            X[ii * LD + col] = acc;
        }
        bar_sync(2, prep::kThreads);
        for (int e = tid; e < nel; e += prep::kThreads) {
            const int ii = e / (b * 16), col = e % (b * 16);
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc += Tf[(b * 16 + ii) * LD + b * 16 + m] * X[m * LD + col];
            Tf[(b * 16 + ii) * LD + col] = -acc;
        }
        bar_sync(2, prep::kThreads);
    }
}

__global__ void __launch_bounds__(prep::kThreads, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, TcArgs a) {
    using namespace prep;
    extern __shared__ uint8_t smraw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so that the compiler
    // keeps the shared address space (plain shared loads and stores, not generic ones)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    float* Af = reinterpret_cast<float*>(sm + oAf);
    float* Tf = reinterpret_cast<float*>(sm + oTf);
    float* gcs = reinterpret_cast<float*>(sm + oSc);
    float* bts = gcs + kC;
    float* kinv = gcs + 2 * kC;
    float* qsv = gcs + 3 * kC;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oBar + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long gh = blockIdx.x;  // chunk * H + head
    const int chunk = (int)(gh / a.H), h = (int)(gh % a.H);
    if (chunk >= a.n_chunks[0]) return;
    const int n = a.chunk_seq[chunk];
    long bos, eos;
    seq_bounds(a, n, bos, eos);
    const long t0 = bos + (long)(chunk - a.chunk_first[n]) * kC;
    const int L = (eos - t0 < kC) ? (int)(eos - t0) : kC;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        prefetch_tmap(&mQ);
        prefetch_tmap(&mK);
        prefetch_tmap(&mV);
    }
    if (warp == 0) {
        tmem_alloc(tbase, kTmemCols);
        tmem_relinquish();
    }
    if (tid < kC) {
        const bool in = tid < L;
        gcs[tid] = in ? a.g[(t0 + tid) * a.H + h] : 0.f;
        bts[tid] = in ? a.beta[(t0 + tid) * a.H + h] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], 49152);
        for (int c = 0; c < 2; ++c) {
            tma_load_3d(sm + oKQ + c * 16384, &mK, &bars[0], c * 64, h, (int)t0);
            tma_load_3d(sm + oKQ + c * 16384 + 8192, &mQ, &bars[0], c * 64, h, (int)t0);
            tma_load_3d(sm + oV + c * 8192, &mV, &bars[0], c * 64, h, (int)t0);
        }
    }
    if (warp == 0) {  // inclusive scan of g, two per lane
        const float g0 = gcs[2 * lane], g1 = gcs[2 * lane + 1];
        float s = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += t;
        }
        __syncwarp();
        gcs[2 * lane] = s - g1;
        gcs[2 * lane + 1] = s;
    }
    bool ok = mbar_wait(&bars[0], 0, kPolls);
    if (ok && L < kC) {  // rows past the end of the sequence hold other tokens: zero them
        for (int e = tid; e < (kC - L) * 8 * 5; e += kThreads) {
            const int r = L + e / 40, part = e % 40;  // 5 tiles x 8 chunks of 16 B
            const int tile = part / 8, ch = part % 8;
            uint8_t* base = tile < 2 ? sm + oKQ + tile * 16384 : (tile < 4 ? sm + oKQ + (tile - 2) * 16384 + 8192
                                                                            : nullptr);
            if (tile == 4) {
                *reinterpret_cast<uint4*>(sm + oV + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + oV + 8192 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            } else {
                *reinterpret_cast<uint4*>(base + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        fence_async_smem();
    }
    __syncthreads();
    if (!ok) {
        if (tid == 0) record_error(a.err, GDN_ERR_TIMEOUT);
    } else if (tid == 0) {
        tc_fence_after();
        const uint32_t kq = smem_u32(sm + oKQ);
        for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_bf16_ss(tm, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024),
                        idesc_bf16(128, 128, 0, 0), k > 0);
        }
        mma_commit(&bars[1]);
    }
    ok = ok && mbar_wait(&bars[1], 0, kPolls);
    tc_fence_after();
    if (!ok) {
        if (tid == 0) record_error(a.err, GDN_ERR_TIMEOUT);
    } else {
        // ---- E1: Gram rows -> norms, A (fp32, smem), Aqk (bf16, workspace) ----
        const uint32_t lane_addr = tm + (static_cast<uint32_t>(warp * 32) << 16);
        float row[64];
        {
            uint32_t r0[32], r1[32];
            tmem_ld32(lane_addr + 0, r0);
            tmem_ld32(lane_addr + 32, r1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) { row[j] = __uint_as_float(r0[j]); row[32 + j] = __uint_as_float(r1[j]); }
        }
        float diag = 0.f;
        if (tid < kC) {
#pragma unroll
            for (int j = 0; j < 64; ++j) if (j == tid) diag = row[j];
            kinv[tid] = a.use_l2 ? rsqrtf(diag + kL2Eps) : 1.0f;
        } else {
            uint32_t r2[32], r3[32];
            tmem_ld32(lane_addr + 64, r2);
            tmem_ld32(lane_addr + 96, r3);
            tmem_wait_ld();
            const int ii = tid - kC;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j == ii) diag = __uint_as_float(r2[j]);
                if (j + 32 == ii) diag = __uint_as_float(r3[j]);
            }
            qsv[ii] = a.scale * (a.use_l2 ? rsqrtf(diag + kL2Eps) : 1.0f);
        }
        tc_fence_before();
        __syncthreads();
        if (tid < kC) {
            const int i = tid;
            const float gi = gcs[i], f = bts[i] * kinv[i];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                Af[i * LD + j] = j < i ? f * __expf(gi - gcs[j]) * row[j] * kinv[j] : 0.f;
            // per-token factors for the state pass
            float* sc = a.scal + gh * 4 * kC;
            const float glast = gcs[kC - 1];
            sc[i] = __expf(gi) * qsv[i];
            sc[kC + i] = __expf(glast - gi) * kinv[i];
            sc[2 * kC + i] = gi;
            if (i == 0) sc[3 * kC] = __expf(glast);
        } else {
            const int i = tid - kC;
            const float gi = gcs[i], f = qsv[i];
            uint4* dst = reinterpret_cast<uint4*>(a.Aqk + gh * kC * kC + (long)i * kC);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = c8 * 8 + e;
                    v[e] = j <= i ? f * __expf(gi - gcs[j]) * row[j] * kinv[j] : 0.f;
                }
                dst[c8] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                     pack_bf16x2(v[6], v[7]));
            }
        }
        __syncthreads();
        // ---- T = (I + A)^-1 (the 16 x 48 fp32 scratch of the block steps lives in the T' tile,
        //      which is written only after the inverse is complete) ----
        unit_lower_inverse(Af, Tf, reinterpret_cast<float*>(sm + oTP), tid);
        // ---- T' = T diag(beta e^gc kinv) and T'' = T diag(beta) as bf16 SW128 operand tiles ----
        {
            const int i = tid & 63, which = tid >> 6;
            uint8_t* dst = sm + (which ? oTPP : oTP);
            float v[8];
            for (int c8 = 0; c8 < 8; ++c8) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = c8 * 8 + e;
                    const float cf = which ? bts[j] : bts[j] * __expf(gcs[j]) * kinv[j];
                    v[e] = Tf[i * LD + j] * cf;
                }
                st_sw128_chunk(dst, i, c8, v);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t kq = smem_u32(sm + oKQ), vv = smem_u32(sm + oV);
            const uint32_t tp = smem_u32(sm + oTP), tpp = smem_u32(sm + oTPP);
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tm + 0, sdesc_sw128(kq + k * 2048, 16384, 1024), sdesc_sw128(tp + k * 32, 16, 1024),
                            idesc_bf16(128, 64, 1, 0), k > 0);
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tm + 64, sdesc_sw128(vv + k * 2048, 8192, 1024), sdesc_sw128(tpp + k * 32, 16, 1024),
                            idesc_bf16(128, 64, 1, 0), k > 0);
            mma_commit(&bars[1]);
        }
        const bool ok2 = mbar_wait(&bars[1], 1, kPolls);
        tc_fence_after();
        if (!ok2) {
            if (tid == 0) record_error(a.err, GDN_ERR_TIMEOUT);
        } else {
            // ---- E2: W (token-major, staged) and U^T (row per thread) to the workspace ----
            __nv_bfloat16* Wst = reinterpret_cast<__nv_bfloat16*>(sm + oAf);  // 64 x 128 bf16 = 16 KB
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + 0, r0);
                tmem_ld32(lane_addr + 32, r1);
                tmem_wait_ld();
                const int d = tid;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    Wst[i * kD + d] = __float2bfloat16_rn(__uint_as_float(r0[i]));
                    Wst[(32 + i) * kD + d] = __float2bfloat16_rn(__uint_as_float(r1[i]));
                }
            }
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + 64, r0);
                tmem_ld32(lane_addr + 96, r1);
                tmem_wait_ld();
                uint4* dst = reinterpret_cast<uint4*>(a.Ut + gh * kD * kC + (long)tid * kC);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    dst[c8] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c8]), __uint_as_float(r0[8 * c8 + 1])),
                                         pack_bf16x2(__uint_as_float(r0[8 * c8 + 2]), __uint_as_float(r0[8 * c8 + 3])),
                                         pack_bf16x2(__uint_as_float(r0[8 * c8 + 4]), __uint_as_float(r0[8 * c8 + 5])),
                                         pack_bf16x2(__uint_as_float(r0[8 * c8 + 6]), __uint_as_float(r0[8 * c8 + 7])));
                    dst[4 + c8] = make_uint4(pack_bf16x2(__uint_as_float(r1[8 * c8]), __uint_as_float(r1[8 * c8 + 1])),
                                             pack_bf16x2(__uint_as_float(r1[8 * c8 + 2]), __uint_as_float(r1[8 * c8 + 3])),
                                             pack_bf16x2(__uint_as_float(r1[8 * c8 + 4]), __uint_as_float(r1[8 * c8 + 5])),
                                             pack_bf16x2(__uint_as_float(r1[8 * c8 + 6]), __uint_as_float(r1[8 * c8 + 7])));
                }
            }
            __syncthreads();
            const uint4* src = reinterpret_cast<const uint4*>(Wst);
            uint4* dst = reinterpret_cast<uint4*>(a.W + gh * kC * kD);
            for (int e = tid; e < kC * kD / 8; e += kThreads) dst[e] = src[e];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// ---- 3. serial state pass ------------------------------------------------------------------------

namespace st {
constexpr int kThreads = 384;               // 12 warps = 3 warpgroups
// register split: launched at 168 per thread (384 x 168 = 64512); the producer / MMA warpgroup
// gives back down to 80 and the two epilogue warpgroups rise to 208: 128 x 80 + 256 x 208 = 63488
constexpr int kRegsLow = 80, kRegsHigh = 208;
constexpr uint32_t oS = 0;                  // S bf16 operand: 2 atom columns x 128 rows = 32 KB
constexpr uint32_t oA1 = 32768;             // V_new^T bf16 [128 x 64] SW128 = 16 KB
constexpr uint32_t oA2 = 49152;             // V_new^T diag(kfac) = 16 KB
constexpr uint32_t oStage = 65536;          // two stages
// stage layout
constexpr uint32_t sWQ = 0;                 // 2 atom columns x (W rows 0-63, Q rows 64-127) = 32 KB
constexpr uint32_t sK = 32768;              // 2 atom columns x 64 rows = 16 KB
constexpr uint32_t sAqk = 49152;            // 64 x 64 = 8 KB
constexpr uint32_t sScal = 57344;           // 4 x 64 fp32 = 1 KB
constexpr uint32_t kStage = 58368;          // multiple of 1024
constexpr uint32_t oOt = oStage + 2 * kStage;    // output tile fp32 [64 tokens][128] = 32 KB
constexpr uint32_t oQs = oOt + 32768;            // output row factors of the current chunk (64 fp32)
constexpr uint32_t oBar = oQs + 256;
constexpr uint32_t kBytes = oBar + 256;
constexpr uint32_t kSmem = kBytes + 1024;
constexpr uint32_t kStageTx = 32768 + 16384 + 8192 + 1024;
// barriers
enum { FULL0 = 0, FULL1, EMPTY0, EMPTY1, SBF, DA1, A12, SFULL, DA2_0, DA2_1, DO_0, DO_1, DAE_0, DAE_1, NBAR };
constexpr uint32_t kTmemCols = 512;
}  // namespace st

__global__ void __launch_bounds__(st::kThreads, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mAqk, TcArgs a) {
    using namespace st;
    extern __shared__ uint8_t smraw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so that the compiler
    // keeps the shared address space (plain shared loads and stores, not generic ones)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oBar + 8 * NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oBar + 8 * NBAR + 4);
    float* otile = reinterpret_cast<float*>(sm + oOt);
    float* qs_s = reinterpret_cast<float*>(sm + oQs);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int n = unit / a.H, h = unit % a.H;
    long bos, eos;
    if (!seq_bounds(a, n, bos, eos)) return;  // reported by the chunk map kernel
    const int nck = (int)((eos - bos + kC - 1) / kC);
    const int first = a.chunk_first[n];

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == EMPTY0 || i == EMPTY1) cnt = 2;  // MMA commit + state epilogue
            mbar_init(&bars[i], cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tbase, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    const uint32_t tS = tm, tDA0 = tm + 128, tDO0 = tm + 384;

    auto stage_ptr = [&](int s) { return sm + oStage + s * kStage; };
    auto fail = [&]() {
        record_error(a.err, GDN_ERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp < 4) {
    reg_dealloc<kRegsLow>();
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            for (int c = 0; c < nck; ++c) {
                const int s = c & 1;
                if (c >= 2 && !mbar_wait(&bars[EMPTY0 + s], ((c >> 1) - 1) & 1, kPolls)) { fail(); break; }
                if (*abort_flag) break;
                uint8_t* sp = stage_ptr(s);
                const long gh = (long)(first + c) * a.H + h;
                const int t0 = (int)(bos + (long)c * kC);
                mbar_arrive_expect_tx(&bars[FULL0 + s], kStageTx);
                for (int ac = 0; ac < 2; ++ac) {
                    tma_load_2d(sp + sWQ + ac * 16384, &mW, &bars[FULL0 + s], ac * 64, (int)(gh * kC));
                    tma_load_3d(sp + sWQ + ac * 16384 + 8192, &mQ, &bars[FULL0 + s], ac * 64, h, t0);
                    tma_load_3d(sp + sK + ac * 8192, &mK, &bars[FULL0 + s], ac * 64, h, t0);
                }
                tma_load_2d(sp + sAqk, &mAqk, &bars[FULL0 + s], 0, (int)(gh * kC));
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                    ::"r"(smem_u32(sp + sScal)), "l"(a.scal + gh * 4 * kC), "r"(1024u), "r"(smem_u32(&bars[FULL0 + s]))
                    : "memory");
            }
            // drain: wait until the last issued stages have landed before the CTA may exit
            for (int c = max(0, nck - 2); c < nck; ++c) mbar_wait(&bars[FULL0 + (c & 1)], (c >> 1) & 1, kPolls);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            // descriptors: the K step adds (bytes >> 4) to the start-address field
            const uint64_t dS = sdesc_sw128(smem_u32(sm + oS), 16, 1024);
            const uint64_t dA1 = sdesc_sw128(smem_u32(sm + oA1), 16, 1024);
            const uint64_t dA2 = sdesc_sw128(smem_u32(sm + oA2), 16, 1024);
            const uint64_t dStage0 = sdesc_sw128(smem_u32(stage_ptr(0)), 16, 1024);
            const uint64_t dStageK0 = sdesc_sw128(smem_u32(stage_ptr(0) + sK), 8192, 1024);
            constexpr uint32_t kIdA = idesc_bf16(128, 64, 0, 0), kIdS = idesc_bf16(128, 128, 0, 1);
            for (int c = 0; c < nck; ++c) {
                const int s = c & 1, b = c & 1;
                const uint64_t dSt = dStage0 + (uint64_t)((s * kStage) >> 4);
                const uint64_t dK = dStageK0 + (uint64_t)((s * kStage) >> 4);
                if (!mbar_wait(&bars[FULL0 + s], (c >> 1) & 1, kPolls)) { fail(); break; }
                if (!mbar_wait(&bars[SBF], c & 1, kPolls)) { fail(); break; }
                if (c >= 2 && !mbar_wait(&bars[DAE_0 + b], ((c >> 1) - 1) & 1, kPolls)) { fail(); break; }
                if (*abort_flag) break;
                tc_fence_after();
                const uint32_t tDA = tDA0 + b * 128, tDO = tDO0 + b * 64;
                // S [W;Q]^T, W part first (the serial chain needs it)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                    mma_bf16_ss(tDA, dS + off, dSt + sWQ / 16 + off, kIdA, k > 0);
                }
                mma_commit(&bars[DA1]);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                    mma_bf16_ss(tDA + 64, dS + off, dSt + (sWQ + 8192) / 16 + off, kIdA, k > 0);
                }
                mma_commit(&bars[DA2_0 + b]);
                if (!mbar_wait(&bars[A12], c & 1, kPolls)) { fail(); break; }
                tc_fence_after();
                // S += (V_new^T diag(kfac)) K      (K is the MN-major B operand)
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_bf16_ss(tS, dA2 + k * 2, dK + k * 128, kIdS, 1);
                mma_commit(&bars[SFULL]);
                // O_intra^T = V_new^T Aqk^T
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_bf16_ss(tDO, dA1 + k * 2, dSt + sAqk / 16 + k * 2, kIdA, k > 0);
                mma_commit(&bars[DO_0 + b]);
                mma_commit(&bars[EMPTY0 + s]);
            }
        }
    }  // warps 2-3: idle
    } else {
    reg_alloc<kRegsHigh>();
    if (warp < 8) {
        // ================= state epilogue (serial chain) =================
        const int q4 = warp & 3;               // TMEM lane quarter
        const int r = q4 * 32 + lane;          // state row (d_v index) = TMEM lane
        const uint32_t lrow = static_cast<uint32_t>(q4 * 32) << 16;
        uint8_t* Sb = sm + oS;
        // initial state: S_bf16 <- S0, TMEM S <- gamma_0 S0 (32 columns at a time)
        {
            const float* src = a.initial_state ? a.initial_state + ((long)unit * kD + r) * kD : nullptr;
            float* dst = (nck == 0 && a.final_state) ? a.final_state + ((long)unit * kD + r) * kD : nullptr;
            float g0 = 0.f;
            if (nck > 0) {
                if (mbar_wait(&bars[FULL0], 0, kPolls)) g0 = reinterpret_cast<const float*>(stage_ptr(0) + sScal)[3 * kC];
                else fail();
            }
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float4 t = src ? *reinterpret_cast<const float4*>(src + blk * 32 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    f[j] = t.x; f[j + 1] = t.y; f[j + 2] = t.z; f[j + 3] = t.w;
                }
                if (nck == 0) {
                    if (dst)
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(dst + blk * 32 + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                    continue;
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_sw128_chunk(Sb + (blk >> 1) * 16384, r, (blk & 1) * 4 + c8, f + 8 * c8);
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(g0 * f[j]);
                tmem_st32(tS + lrow + blk * 32, v);
            }
            if (nck > 0) {
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                bar_sync(1, 128);
                if (r == 0) mbar_arrive(&bars[SBF]);
            }
        }
        uint4 up_next[8];
        if (nck > 0) {
            const uint4* src = reinterpret_cast<const uint4*>(a.Ut + ((long)first * a.H + h) * kD * kC + (long)r * kC);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) up_next[c8] = __ldg(src + c8);
        }
        for (int c = 0; c < nck; ++c) {
            const int s = c & 1, b = c & 1;
            const uint8_t* sp = stage_ptr(s);
            const float* scal = reinterpret_cast<const float*>(sp + sScal);
            const long gh = (long)(first + c) * a.H + h;
            const bool last = (c + 1 == nck);
            // U^T row r comes straight from the workspace, loaded one chunk ahead; so does the next
            // chunk's decay
            uint4 up[8];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) up[c8] = up_next[c8];
            const float gnext = last ? 1.0f : __ldg(a.scal + (gh + a.H) * 4 * kC + 3 * kC);
            if (!last) {
                const uint4* src = reinterpret_cast<const uint4*>(a.Ut + (gh + a.H) * kD * kC + (long)r * kC);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) up_next[c8] = __ldg(src + c8);
            }
            if (!mbar_wait(&bars[DA1], c & 1, kPolls)) { fail(); break; }
            tc_fence_after();
            // ---- V_new^T row r = U^T row r - (S W^T) row r, 32 tokens at a time ----
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t v[32];
                tmem_ld32(tDA0 + b * 128 + lrow + 32 * hf, v);
                tmem_wait_ld();
                float u[32];
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const uint4 q = up[4 * hf + c8];
                    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
                        u[8 * c8 + 2 * e] = f.x - __uint_as_float(v[8 * c8 + 2 * e]);
                        u[8 * c8 + 2 * e + 1] = f.y - __uint_as_float(v[8 * c8 + 2 * e + 1]);
                    }
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_sw128_chunk(sm + oA1, r, 4 * hf + c8, u + 8 * c8);
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] *= scal[kC + 32 * hf + i];
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_sw128_chunk(sm + oA2, r, 4 * hf + c8, u + 8 * c8);
            }
            fence_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (r == 0) {
                mbar_arrive(&bars[A12]);
                mbar_arrive(&bars[EMPTY0 + s]);
            }
            if (!mbar_wait(&bars[SFULL], c & 1, kPolls)) { fail(); break; }
            tc_fence_after();
            // ---- S: mirror as bf16 operand, pre-decay by the next chunk's gamma ----
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t v[32];
                tmem_ld32(tS + lrow + blk * 32, v);
                tmem_wait_ld();
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                if (last) {
                    if (a.final_state) {
                        float* dst = a.final_state + ((long)unit * kD + r) * kD + blk * 32;
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(dst + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                    }
                } else {
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        st_sw128_chunk(Sb + (blk >> 1) * 16384, r, (blk & 1) * 4 + c8, f + 8 * c8);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(gnext * f[j]);
                    tmem_st32(tS + lrow + blk * 32, v);
                }
            }
            if (!last) {
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                bar_sync(1, 128);
                if (r == 0) mbar_arrive(&bars[SBF]);
            }
        }
    } else {
        // ================= output epilogue (O and the gate) =================
        // Phase 1 (thread = column r = TMEM lane): o[r][i] = qsc_i (Q S^T)[i][r] + (Aqk V_new)[i][r]
        // into the fp32 tile otile[i][r].  Phase 2 (warp = token row): RMS over the row, gate with
        // z, vectorised stores.  Reads nothing from the operand ring, so it never holds it up.
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int wq = warp - 8;               // 0..3 within the group
        const uint32_t lrow = static_cast<uint32_t>(q4 * 32) << 16;
        const long tok_stride = (long)a.H * kD;
        float4 w4 = make_float4(1.f, 1.f, 1.f, 1.f);
        if (a.w) w4 = *reinterpret_cast<const float4*>(a.w + 4 * lane);
        float qa_n = 0.f, qb_n = 0.f;
        float4 zf_n[kC / 4];
        auto og_prefetch = [&](int cn) {
            const long ghn = (long)(first + cn) * a.H + h;
            const long tn = bos + (long)cn * kC;
            const int Ln = (eos - tn < kC) ? (int)(eos - tn) : kC;
            if (wq == 0) {
                qa_n = __ldg(a.scal + ghn * 4 * kC + lane);
                qb_n = __ldg(a.scal + ghn * 4 * kC + 32 + lane);
            }
#pragma unroll
            for (int m = 0; m < kC / 4; ++m) {
                const int i = wq + 4 * m;
                zf_n[m] = (a.z && i < Ln)
                              ? __ldg(reinterpret_cast<const float4*>(a.z + (tn + i) * tok_stride + (long)h * kD) + lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        if (nck > 0) og_prefetch(0);
        for (int c = 0; c < nck; ++c) {
            const int b = c & 1;
            const long t0 = bos + (long)c * kC;
            const int L = (eos - t0 < kC) ? (int)(eos - t0) : kC;
            const long gh = (long)(first + c) * a.H + h;
            (void)gh;
            // this chunk's row factors and z rows were loaded one chunk ago; start the next chunk's
            const float qa = qa_n, qb = qb_n;
            float4 zf[kC / 4];
#pragma unroll
            for (int m = 0; m < kC / 4; ++m) zf[m] = zf_n[m];
            if (c + 1 < nck) og_prefetch(c + 1);
            if (!mbar_wait(&bars[DA2_0 + b], (c >> 1) & 1, kPolls)) { fail(); break; }
            if (!mbar_wait(&bars[DO_0 + b], (c >> 1) & 1, kPolls)) { fail(); break; }
            tc_fence_after();
            if (wq == 0) {
                qs_s[lane] = qa;
                qs_s[32 + lane] = qb;
            }
            bar_sync(4, 128);                  // qs_s of this chunk is visible
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t p[32], q[32];
                tmem_ld32(tDA0 + b * 128 + 64 + 32 * hf + lrow, p);
                tmem_ld32(tDO0 + b * 64 + 32 * hf + lrow, q);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    otile[(32 * hf + i) * kD + r] = qs_s[32 * hf + i] * __uint_as_float(p[i]) + __uint_as_float(q[i]);
            }
            tc_fence_before();
            bar_sync(4, 128);
            if (r == 0) mbar_arrive(&bars[DAE_0 + b]);
#pragma unroll
            for (int m = 0; m < kC / 4; ++m) {
                const int i = wq + 4 * m;
                const float4 o = *reinterpret_cast<const float4*>(otile + i * kD + 4 * lane);
                float4 res = o;
                if (a.z) {
                    float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
                    ss = warp_sum(ss);
                    const float rinv = rsqrtf(ss / kD + a.eps);
                    const float4 z = zf[m];
                    res.x = w4.x * o.x * rinv * z.x * fast_sigmoid(z.x);
                    res.y = w4.y * o.y * rinv * z.y * fast_sigmoid(z.y);
                    res.z = w4.z * o.z * rinv * z.z * fast_sigmoid(z.z);
                    res.w = w4.w * o.w * rinv * z.w * fast_sigmoid(z.w);
                }
                const long off = (t0 + i) * tok_stride + (long)h * kD + 4 * lane;
                if (i >= L) continue;
                if (a.out_dtype == GDN_BF16) {
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + off) =
                        make_uint2(pack_bf16x2(res.x, res.y), pack_bf16x2(res.z, res.w));
                } else {
                    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + off) = res;
                }
            }
            bar_sync(4, 128);                  // otile and qs_s are reused by the next chunk
        }
    }
    }  // epilogue warpgroups
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// ---- host side -----------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool map_tokens(CUtensorMap* m, const void* base, int total_T, int H) {
    // [total_T, H, 128] bf16 -> dims (128, H, total_T), box (64, 1, 64), 128-byte swizzle
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return get_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_rows(CUtensorMap* m, const void* base, long rows, int cols, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return get_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_tc_workspace_bytes(int num_seqs, int total_T, int H) {
    return ws_layout(num_seqs, total_T, H).total;
}

bool prefill_tc_supported(const PrefillArgs& a) {
    return a.d == 128 && a.qkv_dtype == GDN_BF16 && get_encoder() != nullptr && a.total_T > 0;
}

cudaError_t launch_prefill_tc(const PrefillArgs& p, cudaStream_t s) {
    const WsLayout L = ws_layout(p.num_seqs, p.total_T, p.H);
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    TcArgs a{};
    a.cu = p.cu_seqlens; a.num_seqs = p.num_seqs; a.total_T = p.total_T; a.H = p.H;
    a.g = p.g; a.beta = p.beta; a.scale = p.scale; a.use_l2 = p.use_l2;
    a.chunk_seq = reinterpret_cast<int32_t*>(ws + L.off_map);
    a.chunk_first = reinterpret_cast<int32_t*>(ws + L.off_first);
    a.n_chunks = reinterpret_cast<int32_t*>(ws + L.off_count);
    a.W = reinterpret_cast<__nv_bfloat16*>(ws + L.off_W);
    a.Ut = reinterpret_cast<__nv_bfloat16*>(ws + L.off_Ut);
    a.Aqk = reinterpret_cast<__nv_bfloat16*>(ws + L.off_Aqk);
    a.scal = reinterpret_cast<float*>(ws + L.off_scal);
    a.initial_state = p.initial_state; a.final_state = p.final_state;
    a.z = p.z; a.w = p.w; a.eps = p.eps; a.out = p.out; a.out_dtype = p.out_dtype; a.err = p.err;

    CUtensorMap mQ, mK, mV, mW, mAqk;
    if (!map_tokens(&mQ, p.q, p.total_T, p.H) || !map_tokens(&mK, p.k, p.total_T, p.H) ||
        !map_tokens(&mV, p.v, p.total_T, p.H) || !map_rows(&mW, a.W, L.nch * kC, kD, 64) ||
        !map_rows(&mAqk, a.Aqk, L.nch * kC, kC, 64))
        return cudaErrorInvalidValue;

    chunk_map_kernel<<<1, 1024, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep::kSmem);
    if (e != cudaSuccess) return e;
    chunk_prep_kernel<<<(unsigned)L.nch, prep::kThreads, prep::kSmem, s>>>(mQ, mK, mV, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st::kSmem);
    if (e != cudaSuccess) return e;
    chunk_state_kernel<<<(unsigned)((long)p.num_seqs * p.H), st::kThreads, st::kSmem, s>>>(mQ, mK, mW, mAqk, a);
    return cudaGetLastError();
}

}  // namespace gdn
