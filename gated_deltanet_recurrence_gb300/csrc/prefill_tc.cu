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
// Launches on the caller's stream:
//   chunk_map_kernel    numbers the chunks of all sequences (varlen) in the workspace, and ranks the
//                       sequences by length for the serial pass.
//   then either (few (sequence, head) units: at most half the SMs)
//   chunk_fused_kernel  one cooperative launch, one CTA per SM: CTAs 0 .. units-1 run the serial
//                       pass, the others prepare chunks (three at a time) and publish each by a
//                       ready flag the serial pass acquires;
//   or
//   chunk_prep_kernel   one CTA per (chunk, head), all in parallel: TMA loads of K, Q, V; one MMA
//                       [K;Q][K;Q]^T (M=128, N=128, K=128); the triangular solve on the CUDA
//                       cores; two MMAs W^T = K^T T'^T and U^T = V^T T''^T (MN-major A from the
//                       same K / V tiles); W, U^T, Aqk, the scaled rows Q~ and K~ (bf16) and
//                       per-token factors to the workspace;
//   chunk_state_kernel  one CTA per (sequence, head), walking the chunks in order, warp-specialised:
//                       warp 0 issues TMA loads of the next chunk's operands (two-stage ring),
//                       warp 1 issues the MMAs (warps 0-3 run with few registers), warps 4-7 run
//                       the state epilogue (the serial chain: V_new, then S), warps 8-11 and 12-15
//                       the output epilogue of alternate chunks (O and the fused RMSNorm * SiLU
//                       gate).  The state S is fp32 in TMEM (lanes = rows d_v, columns = d_k) and
//                       is mirrored as a bf16 operand tile in shared memory.
//   TMEM per state CTA: S [0,128), two buffers of S W^T [128,256), two of O (tokens as rows) [256,512).
//
// Every mbarrier wait is bounded; on a timeout the kernel records GDN_ERR_TIMEOUT and its roles
// stop issuing work, wait (bounded) for what they issued, free TMEM and return.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_fp16.h>

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
    size_t off_map, off_first, off_count, off_order, off_W, off_Ut, off_Aqk, off_scal, off_Qt, off_Kt, off_gam,
        off_ready, off_Sx, off_Vx, off_oready, total;
    bool exports;      // room for the fused kernel's exported state
};

__host__ __device__ inline long max_chunks(int num_seqs, int total_T) { return (long)total_T / kC + num_seqs; }

inline WsLayout ws_layout(int num_seqs, int total_T, int H, bool exports) {
    WsLayout w{};
    w.exports = exports;
    const long mc = max_chunks(num_seqs, total_T);
    w.nch = mc * H;
    auto al = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    size_t o = 0;
    w.off_map = o;   o = al(o + sizeof(int32_t) * mc);               // chunk -> sequence
    w.off_first = o; o = al(o + sizeof(int32_t) * (num_seqs + 1));   // first chunk of each sequence
    w.off_count = o; o = al(o + sizeof(int32_t) * 4);                 // number of chunks
    w.off_order = o; o = al(o + sizeof(int32_t) * num_seqs);          // sequences, most chunks first
    w.off_W = o;     o = al(o + sizeof(__nv_bfloat16) * w.nch * kC * kD);
    w.off_Ut = o;    o = al(o + sizeof(__nv_bfloat16) * w.nch * kD * kC);
    w.off_Aqk = o;   o = al(o + sizeof(__nv_bfloat16) * w.nch * kC * kC);
    w.off_scal = o;  o = al(o + sizeof(float) * w.nch * 4 * kC);
    w.off_Qt = o;    o = al(o + sizeof(__nv_bfloat16) * w.nch * kC * kD);   // diag(e^gc qs) Q
    w.off_Kt = o;    o = al(o + sizeof(__nv_bfloat16) * w.nch * kC * kD);   // diag(e^(glast-gc) kinv) K
    w.off_gam = o;   o = al(o + sizeof(float) * w.nch * kD);                // per-channel e^(gc_last)
    w.off_ready = o; o = al(o + sizeof(int32_t) * w.nch);                  // fused kernel: chunk ready flags
    if (exports) {  // fused kernel, export form: state tile, V_new^T, flag per chunk-head slot
        w.off_Sx = o;     o = al(o + (size_t)32768 * w.nch);
        w.off_Vx = o;     o = al(o + (size_t)16384 * w.nch);
        w.off_oready = o; o = al(o + sizeof(int32_t) * w.nch);
    }
    w.total = o;
    return w;
}

struct TcArgs {
    const int32_t* cu;   // may be null: fixed length
    int num_seqs, total_T, H, Hk;
    int d;               // head size of the caller's tensors (64 or 128); tiles are 128 wide, the
                         // columns past d are zeros (TMA fills them) and stay zero throughout
    const __nv_bfloat16* q;  // raw q, k [total_T, Hk, 128] and v [total_T, H, 128]: convolution history
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    ConvArgs conv;
    const float* g;
    const float* beta;
    float scale;
    int use_l2;
    int32_t* chunk_seq;
    int32_t* chunk_first;
    int32_t* n_chunks;
    int32_t* seq_order;  // sequences by decreasing chunk count (the two-kernel serial pass runs them in it)
    __nv_bfloat16* W;
    __nv_bfloat16* Ut;
    __nv_bfloat16* Aqk;
    float* scal;
    __nv_bfloat16* Qt;
    __nv_bfloat16* Kt;
    float* gam;          // decay per key channel: e^(gc_last) per chunk and channel [nch][128]
    int32_t* ready;      // fused kernel only: per chunk-head slot, 1 once its entries are written
    // fused kernel with exported state (null otherwise): per chunk-head slot the state at the chunk's
    // start as the serial pass's bf16 operand tile (32 KB, swizzled as in shared memory), V_new^T
    // (16 KB, likewise) and a flag set once both are written
    uint8_t* Sx;
    uint8_t* Vx;
    int32_t* oready;
    long nch;            // chunk-head slots of the workspace
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
    __shared__ int32_t longest;
    const int tid = threadIdx.x;
    if (tid == 0) longest = 0;
    if (a.ready)  // fused kernel: no chunk is ready yet
        for (long i = tid; i < a.nch; i += 1024) a.ready[i] = 0;
    if (a.oready)  // export form: no chunk's state is exported yet
        for (long i = tid; i < a.nch; i += 1024) a.oready[i] = 0;
    // per-thread contiguous block of sequences
    const int per = (a.num_seqs + 1023) / 1024;
    const int s0 = tid * per, s1 = min(a.num_seqs, s0 + per);
    int32_t cnt = 0, mx = 0;
    for (int n = s0; n < s1; ++n) {
        long bos, eos;
        if (seq_bounds(a, n, bos, eos)) {
            const int32_t c = (int32_t)((eos - bos + kC - 1) / kC);
            cnt += c;
            mx = max(mx, c);
        } else {
            record_error(a.err, GDN_ERR_CU_SEQLENS);
        }
    }
    part[tid] = cnt;
    __syncthreads();
    atomicMax(&longest, mx);
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
        a.n_chunks[1] = longest;  // chunks of the longest sequence
        a.n_chunks[2] = 0;        // fused kernel: work counter of the preparing CTAs
        a.n_chunks[3] = 0;        // fused kernel with exported state: output work counter
    }
    // the order in which the serial pass starts the sequences: most chunks first, so that the long
    // chains are not the last to begin (ties by index; more than 1024 sequences keep their order)
    __syncthreads();  // part[] is reused for the chunk counts
    if (a.num_seqs <= 1024) {
        long bos, eos;
        const int32_t c = (tid < a.num_seqs && seq_bounds(a, tid, bos, eos)) ? (int32_t)((eos - bos + kC - 1) / kC) : -1;
        part[tid] = c;
        __syncthreads();
        if (tid < a.num_seqs) {
            int rank = 0;
            for (int m = 0; m < a.num_seqs; ++m) {
                const int32_t cm = part[m];
                rank += (cm > c) || (cm == c && m < tid);
            }
            a.seq_order[rank] = tid;
        }
    } else {
        for (int n = tid; n < a.num_seqs; n += 1024) a.seq_order[n] = n;
    }
}

// ---- shared helpers --------------------------------------------------------------------------------

// SiLU from sigma(x) = (1 + tanh(x / 2)) / 2 with the hardware tanh approximation (relative error
// near 5e-4, below the bf16 rounding that follows wherever it is used):
// x sigma(x) = h + h tanh(h) with h = x / 2.
__device__ __forceinline__ float fast_silu(float x) {
    const float hx = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hx));
    return fmaf(hx, t, hx);
}

// SiLU of two values at once with the packed half-precision tanh (inputs are the gate's z, of order
// one; the result is rounded to the output type right after): x sigma(x) = h + h tanh(h), h = x / 2.
__device__ __forceinline__ float2 fast_silu2(float x0, float x1) {
    const float h0 = 0.5f * x0, h1 = 0.5f * x1;
    __half2 hh = __floats2half2_rn(h0, h1);
    uint32_t t;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<uint32_t*>(&hh)));
    const float2 tf = __half22float2(*reinterpret_cast<__half2*>(&t));
    return make_float2(fmaf(h0, tf.x, h0), fmaf(h1, tf.y, h1));
}

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

// ---- 2. chunk preparation (parallel) ------------------------------------------------------------

namespace prep {
constexpr int kThreads = 128;
constexpr int LDA = kC + 1;  // A (fp32 64x64): odd stride, conflict-free row/column access
constexpr int LD = kC + 4;   // T and the block scratch: rows stay 16-byte aligned for float4 loads
// Three chunks fit on one SM (68 KB of shared memory, 128 TMEM columns, <= 168 registers each).
// Regions are reused as the chunk proceeds:
constexpr uint32_t oKQ = 0;          // 2 atom columns x (K rows 0-63, Q rows 64-127) = 32 KB; once Q
                                     // is no longer read, V is loaded into Q's rows (MN-block stride 16 KB)
constexpr uint32_t oV = oKQ + 8192;  // V's first 64-column half (the second is 16 KB further)
constexpr uint32_t oAf = 32768;      // A (fp32 64 x 65); after the solve T' and T'' (bf16 SW128 64x64,
constexpr uint32_t oTP = oAf;        // 8 KB each); after the W / U^T product the W staging tile
constexpr uint32_t oTPP = oAf + 8192;
constexpr uint32_t oTf = oAf + 16896;             // T (fp32 64 x 68), 1 KB past A
constexpr uint32_t oSc = oTf + 4 * kC * LD;       // gc, beta, kinv, qs (fp32 x 64 each)
constexpr uint32_t oBar = oSc + 4 * 4 * kC;       // 3 mbarriers (K and Q, products, V) + TMEM base
constexpr uint32_t kBytes = oBar + 64;
constexpr uint32_t kSmem = kBytes + 1024;          // + alignment slack
constexpr uint32_t kTmemCols = 128;                // the Gram product, then W^T and U^T
static_assert(3 * kSmem <= 232448, "three chunks per SM");
}  // namespace prep

// C[16 x 16] (+)= P[16 x 16] Q[16 x 16] for one warp: lane l owns row l / 2 and the 8 columns
// 8 (l % 2) .. 8 (l % 2) + 7 of C, kept in registers.  P and Q are fp32 tiles in shared memory
// with row strides LDP and LDQ (LDQ a multiple of 4: each 8-column half row is two 16-byte loads).
template <int LDP, int LDQ>
__device__ __forceinline__ void warp_mm16(const float* P, const float* Q, float (&c)[8], int lane) {
    const int ii = lane >> 1, c0 = (lane & 1) * 8;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float p = P[ii * LDP + k];
        const float4 q0 = *reinterpret_cast<const float4*>(Q + k * LDQ + c0);
        const float4 q1 = *reinterpret_cast<const float4*>(Q + k * LDQ + c0 + 4);
        c[0] = fmaf(p, q0.x, c[0]); c[1] = fmaf(p, q0.y, c[1]); c[2] = fmaf(p, q0.z, c[2]); c[3] = fmaf(p, q0.w, c[3]);
        c[4] = fmaf(p, q1.x, c[4]); c[5] = fmaf(p, q1.y, c[5]); c[6] = fmaf(p, q1.z, c[6]); c[7] = fmaf(p, q1.w, c[7]);
    }
}

// Blocked inverse of the unit lower-triangular 64x64 matrix I + A (A strictly lower, fp32 in Af
// with row stride LDA) into Tf (row stride LD).  The four diagonal 16x16 blocks by forward
// substitution (one warp per block, one lane per column); then block rows 1..3 in order,
// T_bj = -T_bb sum_{k=j}^{b-1} A_bk T_kj, one warp per block (b, j) with the 16x16 products held
// in registers; X is a per-warp 16 x LD scratch (warps 0-2 only: 3 x 16 x 68 x 4 B = 13 KB).
// Element i (0..63) of the 64 values lo[0..31] | hi[0..31], chosen by a tree of selects: a register
// array indexed by a thread-dependent value would be placed in local memory.
__device__ __forceinline__ float pick64(const uint32_t (&lo)[32], const uint32_t (&hi)[32], int i) {
    uint32_t t[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) t[j] = (i & 32) ? hi[j] : lo[j];
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = (i & w) ? t[j + w] : t[j];
    return __uint_as_float(t[0]);
}

// Bounded wait (2 s at the top SM clock) for another CTA of the fused kernel to publish a chunk's
// workspace entries; false when the bound runs out.
__device__ __forceinline__ bool wait_ready(const int32_t* flag) {
    if (ld_acquire_gpu(flag)) return true;
    const long long limit = static_cast<long long>(kPolls) * 21 / 10;
    const long long t0 = clock64();
    while (!ld_acquire_gpu(flag)) {
        __nanosleep(128);
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// The barrier over the 128 threads that process one chunk: named barrier `id` (and id + 1 inside
// the triangular solve).  In chunk_prep_kernel these are all the CTA's threads; in the fused kernel
// one warpgroup, so that two chunks proceed independently in one CTA.
struct GroupBar {
    uint32_t id;
    uint32_t n = 128;  // threads of the group
    __device__ __forceinline__ void sync() const { bar_sync(id, n); }
    __device__ __forceinline__ bool sync_or(bool p) const { return bar_sync_or(id, n, p); }
};

__device__ void unit_lower_inverse(const float* Af, float* Tf, int tid, GroupBar gb) {
    constexpr int LD = prep::LD, LDA = prep::LDA;
    const int warp = tid >> 5, lane = tid & 31;
    {   // diagonal blocks
        const int b0 = warp * 16;
        if (lane < 16) {
            const int jj = lane;
            float t[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int m = 0; m < ii; ++m) {
                    const float v = m >= jj ? Af[(b0 + ii) * LDA + b0 + m] * t[m] : 0.f;
                    if (m & 1) acc1 += v; else acc0 += v;
                }
                t[ii] = ii < jj ? 0.f : (ii == jj ? 1.f : -(acc0 + acc1));
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
    bar_sync(gb.id + 1, prep::kThreads);
    const int ii = lane >> 1, c0 = (lane & 1) * 8;
    for (int b = 1; b < 4; ++b) {
        const int j = warp;  // block column handled by this warp (warps j >= b idle in this row)
        if (j < b) {
            // Y = sum_k A_bk T_kj goes to the block T_bj itself (no other warp reads it in this
            // step), then T_bj = -T_bb Y is formed in registers and written over it
            float* Tbj = Tf + (b * 16) * LD + j * 16;
            float c[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) c[e] = 0.f;
            for (int k = j; k < b; ++k)
                warp_mm16<LDA, LD>(Af + (b * 16) * LDA + k * 16, Tf + (k * 16) * LD + j * 16, c, lane);
#pragma unroll
            for (int e = 0; e < 8; ++e) Tbj[ii * LD + c0 + e] = c[e];
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 8; ++e) c[e] = 0.f;
            warp_mm16<LD, LD>(Tf + (b * 16) * LD + b * 16, Tbj, c, lane);
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 8; ++e) Tbj[ii * LD + c0 + e] = -c[e];
        }
        bar_sync(gb.id + 1, prep::kThreads);
    }
}

__device__ __forceinline__ void unpack_bf16x8(uint4 p, float* f) {
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        f[2 * e] = t.x;
        f[2 * e + 1] = t.y;
    }
}

// Short convolution + SiLU ("因果卷积") of one loaded tile (ten 0: Q, 1: K, 2: V; 128B-swizzled
// bf16), in place, rows 0..L-1 of the chunk starting at token t0, by kT threads.  Thread tid owns 8
// consecutive channels (one 16-byte chunk: c8 = tid % 8 of column half (tid / 8) % 2) and
// kR = 1024 / kT rows (segment tid / 16), so a quarter-warp reads or writes one whole 128-byte row.
// Every thread first captures the three raw rows before its segment (from the tile, or, for the
// first segment, from the sequence in global memory or the carried state); after a barrier it
// reads its raw rows, convolves them and writes them back, so no thread reads a row that another
// one has overwritten.  K and Q sit in the two atom columns of the K / Q region (K rows first);
// V's two atom columns start at kVOff, kVAtom bytes apart.
template <int kT, uint32_t kVOff, uint32_t kVAtom>
__device__ __forceinline__ void conv_tiles(uint8_t* sm, const TcArgs& a, int n, int h, int hk, long bos,
                                           long t0, int L, int tid, GroupBar gb, int ten) {
    constexpr int kR = 1024 / kT;
    const int c8 = tid & 7, half = (tid >> 3) & 1, r0 = (tid >> 4) * kR;
    const int x0 = half * 64 + c8 * 8;
    // ten 0: Q, 1: K, 2: V
    uint8_t* tile = ten == 2 ? sm + kVOff + half * kVAtom : sm + prep::oKQ + half * 16384 + (ten == 1 ? 0 : 8192);
    const int d = a.d;
    const __nv_bfloat16* src = ten == 0 ? a.q + hk * d + x0 : (ten == 1 ? a.k + hk * d + x0 : a.v + (long)h * d + x0);
    const long stride = ten == 2 ? (long)a.H * d : (long)a.Hk * d;
    const int chan = ten == 0 ? hk * d + x0 : (ten == 1 ? a.Hk * d + hk * d + x0 : 2 * a.Hk * d + h * d + x0);
    const bool live = r0 < L && x0 < d;  // columns past the head size hold zeros and stay so
    float hist[3][8];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int r = r0 - 3 + j;
        float* f = hist[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
        if (!live) continue;
        if (r >= 0) {
            unpack_bf16x8(*reinterpret_cast<const uint4*>(tile + sw128_offset(r, c8 * 8)), f);
        } else {
            const long t = t0 + r;
            if (t >= bos) {
                unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(src + t * stride)), f);
            } else if (a.conv.state_in) {
                const float* st = a.conv.state_in + ((long)n * a.conv.dim + chan) * 3 + 3 + (t - bos);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = st[e * 3];
            }
        }
    }
    gb.sync();
    if (!live) return;
    uint4 raw[kR];
#pragma unroll
    for (int i = 0; i < kR; ++i)
        raw[i] = r0 + i < L ? *reinterpret_cast<const uint4*>(tile + sw128_offset(r0 + i, c8 * 8)) : make_uint4(0, 0, 0, 0);
    float4 w[8];
    const float4* w4 = reinterpret_cast<const float4*>(a.conv.w) + chan;
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = __ldg(w4 + e);
    float* h0 = hist[0];
    float* h1 = hist[1];
    float* h2 = hist[2];
#pragma unroll
    for (int i = 0; i < kR; ++i) {
        float x[8];
        unpack_bf16x8(raw[i], x);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float y0 = fast_silu(fmaf(w[e].w, x[e], fmaf(w[e].z, h2[e], fmaf(w[e].y, h1[e], w[e].x * h0[e]))));
            const float y1 = fast_silu(fmaf(w[e + 1].w, x[e + 1],
                                            fmaf(w[e + 1].z, h2[e + 1], fmaf(w[e + 1].y, h1[e + 1], w[e + 1].x * h0[e + 1]))));
            o[e / 2] = pack_bf16x2(y0, y1);
        }
        if (r0 + i < L)
            *reinterpret_cast<uint4*>(tile + sw128_offset(r0 + i, c8 * 8)) = make_uint4(o[0], o[1], o[2], o[3]);
#pragma unroll
        for (int e = 0; e < 8; ++e) { h0[e] = h1[e]; h1[e] = h2[e]; h2[e] = x[e]; }
    }
}


// ---- decay per key channel ("6.6 Gated DeltaNet" 6.6.7): the products on the CUDA cores ------------
//
// With g a vector per token, the in-chunk decays enter the contraction over the key channels:
//     A_ij   = beta_i kinv_i kinv_j  sum_c k_ic k_jc e^(G_ic - G_jc)     (j < i)
//     Aqk_ij = qs_i kinv_j           sum_c q_ic k_jc e^(G_ic - G_jc)     (j <= i)
// with G the per-channel inclusive sums of g down the chunk.  Each thread owns a 4 x 4 block of the
// strictly lower triangle (120 blocks for threads 0-119) and takes its first row r as reference:
// e^(G_i - G_j) = e^(G_i - G_r) e^(G_r - G_j), both factors <= 1 (G does not increase down the
// chunk and j < r <= i), so 8 exponentials per channel serve 16 pairs and nothing overflows.  The
// 16 diagonal 4 x 4 blocks take their 6 exponentials per channel directly; all 128 threads share
// them, 8 channels each, and add their partial sums with shuffles.  The channels are processed in
// two halves of 64 so that the transposed copies fit in the T', T'' and A tiles, which are not yet
// in use.  The same pass writes the state pass's operand rows Q~ = qs diag(e^G) Q and
// K~ = kinv diag(e^(G_last - G)) K, the per-channel e^(G_last), and overwrites the K tile with
// K . e^G, the operand of W = T diag(beta kinv) (K . e^G).
namespace pcx {
constexpr int LDG = 68;                      // G^T row stride (floats): [channel][row], 16-byte rows
constexpr int LDK = 64;                      // K^T, Q^T row stride (bf16): 128 bytes
constexpr uint32_t oGT = prep::oAf;
constexpr uint32_t oKT = oGT + 64 * LDG * 4;
constexpr uint32_t oQT = oKT + 64 * LDK * 2;
constexpr uint32_t kEnd = oQT + 64 * LDK * 2;
static_assert(kEnd <= prep::oSc, "per-channel scratch must end before the per-token scalars");
}  // namespace pcx

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void bf16x4(uint2 w, float* f) {
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

__device__ void pc_products(uint8_t* sm, const TcArgs& a, long gh, int h, long t0, int L, int tid,
                            const float* kinv, const float* qsv, const float* bts, float* Af, float* Tf,
                            GroupBar gb) {
    using namespace prep;
    float* GT = reinterpret_cast<float*>(sm + pcx::oGT);
    __nv_bfloat16* KT = reinterpret_cast<__nv_bfloat16*>(sm + pcx::oKT);
    __nv_bfloat16* QT = reinterpret_cast<__nv_bfloat16*>(sm + pcx::oQT);
    constexpr int LG = pcx::LDG, LK = pcx::LDK;
    constexpr float kLog2e = 1.4426950408889634f;

    const bool off = tid < 120;                  // strictly lower block (I, J), J < I, row by row
    int I = 1, J = tid;
    while (J >= I) { J -= I; ++I; }
    const int i0 = 4 * I, j0 = 4 * J;
    const int dr = 4 * (tid >> 3), cg = tid & 7; // diagonal block at row dr; channels e * 8 + cg

    // accA2[2 r + h] = (acc[r][2 h], acc[r][2 h + 1]): the 4 x 4 block in column pairs, so that the
    // products run on the packed two-wide FMA (each lane rounds as fmaf does)
    float2 accA2[8], accQ2[8];
    float dA[6], dQ[10];
#pragma unroll
    for (int e = 0; e < 8; ++e) { accA2[e] = make_float2(0.f, 0.f); accQ2[e] = make_float2(0.f, 0.f); }
#pragma unroll
    for (int e = 0; e < 6; ++e) dA[e] = 0.f;
#pragma unroll
    for (int e = 0; e < 10; ++e) dQ[e] = 0.f;

    for (int hf = 0; hf < 2; ++hf) {
        // (a) per-channel inclusive sums, in log2 units; e^(G_last) for the state pass
        if (tid < 64) {  // all 64 loads of a channel in flight at once, then the running sum
            const bool chan_in = hf * 64 + tid < a.d;  // padded channels: no decay
            const float* gp = a.g + (t0 * a.H + h) * (long)a.d + hf * 64 + tid;
            const long gs = (long)a.H * a.d;
            float gv[kC];
#pragma unroll
            for (int i = 0; i < kC; ++i) gv[i] = (i < L && chan_in) ? __ldg(gp + i * gs) : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kC; ++i) {
                acc += gv[i];
                GT[tid * LG + i] = acc * kLog2e;
            }
            a.gam[gh * kD + hf * 64 + tid] = ex2_approx(acc * kLog2e);
        }
        gb.sync();
        // (b) raw transposed copies; Q~, K~ rows to the workspace; K . e^G in the K tile
        {
            const int i = tid & 63, hc = tid >> 6;
            uint8_t* ktile = sm + oKQ + hf * 16384;
            const uint8_t* qtile = ktile + 8192;
            const float fq = qsv[i], fk = kinv[i];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c8 = hc * 4 + cc;
                const uint4 kr = *reinterpret_cast<const uint4*>(ktile + sw128_offset(i, c8 * 8));
                const uint4 qr = *reinterpret_cast<const uint4*>(qtile + sw128_offset(i, c8 * 8));
                float kf[8], qf[8], qo[8], ko[8], ke[8];
                unpack_bf16x8(kr, kf);
                unpack_bf16x8(qr, qf);
                const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kr);
                const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(&qr);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int cl = c8 * 8 + e;
                    KT[cl * LK + i] = kb[e];
                    QT[cl * LK + i] = qb[e];
                    const float G = GT[cl * LG + i], Gl = GT[cl * LG + kC - 1];
                    const float eg = ex2_approx(G), el = ex2_approx(Gl - G);
                    qo[e] = qf[e] * eg * fq;
                    ko[e] = kf[e] * el * fk;
                    ke[e] = kf[e] * eg;
                }
                *reinterpret_cast<uint4*>(ktile + sw128_offset(i, c8 * 8)) = pack_bf16x8(ke);
                const long ro = gh * kC * kD + (long)i * kD + hf * 64 + c8 * 8;
                *reinterpret_cast<uint4*>(a.Qt + ro) = pack_bf16x8(qo);
                *reinterpret_cast<uint4*>(a.Kt + ro) = pack_bf16x8(ko);
            }
        }
        gb.sync();
        // (c) products over this half's 64 channels
        if (off) {
#pragma unroll 4
            for (int cl = 0; cl < 64; ++cl) {
                const float4 Gi = *reinterpret_cast<const float4*>(GT + cl * LG + i0);
                const float4 Gj = *reinterpret_cast<const float4*>(GT + cl * LG + j0);
                float ki[4], qi[4], kj[4];
                bf16x4(*reinterpret_cast<const uint2*>(KT + cl * LK + i0), ki);
                bf16x4(*reinterpret_cast<const uint2*>(QT + cl * LK + i0), qi);
                bf16x4(*reinterpret_cast<const uint2*>(KT + cl * LK + j0), kj);
                const float ei[4] = {1.f, ex2_approx(Gi.y - Gi.x), ex2_approx(Gi.z - Gi.x), ex2_approx(Gi.w - Gi.x)};
                const float ej[4] = {ex2_approx(Gi.x - Gj.x), ex2_approx(Gi.x - Gj.y), ex2_approx(Gi.x - Gj.z),
                                     ex2_approx(Gi.x - Gj.w)};
                const float2 kje01 = __fmul2_rn(make_float2(kj[0], kj[1]), make_float2(ej[0], ej[1]));
                const float2 kje23 = __fmul2_rn(make_float2(kj[2], kj[3]), make_float2(ej[2], ej[3]));
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float2 e = __fmul2_rn(make_float2(ki[r], qi[r]), make_float2(ei[r], ei[r]));  // (k, q) . e_i
                    const float2 kk = make_float2(e.x, e.x), qq = make_float2(e.y, e.y);
                    accA2[2 * r] = __ffma2_rn(kk, kje01, accA2[2 * r]);
                    accA2[2 * r + 1] = __ffma2_rn(kk, kje23, accA2[2 * r + 1]);
                    accQ2[2 * r] = __ffma2_rn(qq, kje01, accQ2[2 * r]);
                    accQ2[2 * r + 1] = __ffma2_rn(qq, kje23, accQ2[2 * r + 1]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int cl = e * 8 + cg;
            const float4 G = *reinterpret_cast<const float4*>(GT + cl * LG + dr);
            float k[4], q[4];
            bf16x4(*reinterpret_cast<const uint2*>(KT + cl * LK + dr), k);
            bf16x4(*reinterpret_cast<const uint2*>(QT + cl * LK + dr), q);
            const float e10 = ex2_approx(G.y - G.x), e20 = ex2_approx(G.z - G.x), e30 = ex2_approx(G.w - G.x);
            const float e21 = ex2_approx(G.z - G.y), e31 = ex2_approx(G.w - G.y), e32 = ex2_approx(G.w - G.z);
            const float k10 = k[0] * e10, k20 = k[0] * e20, k30 = k[0] * e30;
            const float k21 = k[1] * e21, k31 = k[1] * e31, k32 = k[2] * e32;
            dA[0] = fmaf(k[1], k10, dA[0]); dA[1] = fmaf(k[2], k20, dA[1]); dA[2] = fmaf(k[3], k30, dA[2]);
            dA[3] = fmaf(k[2], k21, dA[3]); dA[4] = fmaf(k[3], k31, dA[4]); dA[5] = fmaf(k[3], k32, dA[5]);
            dQ[0] = fmaf(q[0], k[0], dQ[0]); dQ[1] = fmaf(q[1], k10, dQ[1]); dQ[2] = fmaf(q[1], k[1], dQ[2]);
            dQ[3] = fmaf(q[2], k20, dQ[3]); dQ[4] = fmaf(q[2], k21, dQ[4]); dQ[5] = fmaf(q[2], k[2], dQ[5]);
            dQ[6] = fmaf(q[3], k30, dQ[6]); dQ[7] = fmaf(q[3], k31, dQ[7]); dQ[8] = fmaf(q[3], k32, dQ[8]);
            dQ[9] = fmaf(q[3], k[3], dQ[9]);
        }
        gb.sync();
    }
    // diagonal blocks: sum the 8 channel groups (lanes 8m .. 8m + 7 of one warp)
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
        for (int e = 0; e < 6; ++e) dA[e] += __shfl_xor_sync(0xffffffffu, dA[e], o);
#pragma unroll
        for (int e = 0; e < 10; ++e) dQ[e] += __shfl_xor_sync(0xffffffffu, dQ[e], o);
    }
    // A (fp32) into Af; the decayed Q K^T (fp32) staged in Tf
    if (off) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = i0 + r, j = j0 + b;
                const float2 pa = accA2[2 * r + (b >> 1)], pq = accQ2[2 * r + (b >> 1)];
                Af[i * LDA + j] = bts[i] * kinv[i] * kinv[j] * ((b & 1) ? pa.y : pa.x);
                Tf[i * LD + j] = qsv[i] * kinv[j] * ((b & 1) ? pq.y : pq.x);
            }
    }
    if (cg == 0) {
        const int ia[6] = {1, 2, 3, 2, 3, 3}, ja[6] = {0, 0, 0, 1, 1, 2};
        const int iq[10] = {0, 1, 1, 2, 2, 2, 3, 3, 3, 3}, jq[10] = {0, 0, 1, 0, 1, 2, 0, 1, 2, 3};
#pragma unroll
        for (int e = 0; e < 6; ++e) {
            const int i = dr + ia[e], j = dr + ja[e];
            Af[i * LDA + j] = bts[i] * kinv[i] * kinv[j] * dA[e];
        }
#pragma unroll
        for (int e = 0; e < 10; ++e) {
            const int i = dr + iq[e], j = dr + jq[e];
            Tf[i * LD + j] = qsv[i] * kinv[j] * dQ[e];
        }
    }
    gb.sync();
    if (tid >= kC) {  // decayed Q K^T rows to the workspace, zero above the diagonal
        const int i = tid - kC;
        uint4* dst = reinterpret_cast<uint4*>(a.Aqk + gh * kC * kC + (long)i * kC);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = c8 * 8 + e;
                v[e] = j <= i ? Tf[i * LD + j] : 0.f;
            }
            dst[c8] = pack_bf16x8(v);
        }
    }
}

// One chunk of one head with a decay per key channel (prep2_chunk handles a decay per head):
// everything the state pass needs from it, written to the workspace.  The 128 threads (tid 0..127) synchronise with `gb`; `sm` is this chunk's 1024-aligned shared region,
// `tm` its 256 TMEM columns, `bars` its two mbarriers, the TMA barrier expected at `tma_parity`.
template <bool PC>
__device__ __forceinline__ void prep_chunk(uint8_t* sm, uint32_t tm, uint64_t* bars, uint32_t tma_parity,
                                           GroupBar gb, int tid, long gh, const CUtensorMap* mQ,
                                           const CUtensorMap* mK, const CUtensorMap* mV, const TcArgs& a) {
    using namespace prep;
    float* Af = reinterpret_cast<float*>(sm + oAf);
    float* Tf = reinterpret_cast<float*>(sm + oTf);
    float* gcs = reinterpret_cast<float*>(sm + oSc);
    float* bts = gcs + kC;
    float* kinv = gcs + 2 * kC;
    float* qsv = gcs + 3 * kC;
    const int warp = tid >> 5, lane = tid & 31;
    const int chunk = (int)(gh / a.H), h = (int)(gh % a.H);  // gh = chunk * H + head
    const int hk = h / (a.H / a.Hk);  // query/key head read by value head h
    const int n = a.chunk_seq[chunk];
    long bos, eos;
    seq_bounds(a, n, bos, eos);
    const long t0 = bos + (long)(chunk - a.chunk_first[n]) * kC;
    const int L = (eos - t0 < kC) ? (int)(eos - t0) : kC;

    if (tid < kC) {
        const bool in = tid < L;
        gcs[tid] = (in && !PC) ? a.g[(t0 + tid) * a.H + h] : 0.f;  // per channel: zero here
        bts[tid] = in ? a.beta[(t0 + tid) * a.H + h] : 0.f;
    }
    tc_fence_before();
    gb.sync();
    tc_fence_after();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], 32768);
        for (int c = 0; c < 2; ++c) {
            tma_load_3d(sm + oKQ + c * 16384, mK, &bars[0], c * 64, hk, (int)t0);
            tma_load_3d(sm + oKQ + c * 16384 + 8192, mQ, &bars[0], c * 64, hk, (int)t0);
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
    bool ok = mbar_wait(&bars[0], tma_parity, kPolls);
    if (a.conv.w) {  // fused short convolution of the loaded rows (group-uniform: has barriers)
        if (!gb.sync_or(!ok)) {
            conv_tiles<prep::kThreads, prep::oV, 16384>(sm, a, n, h, hk, bos, t0, L, tid, gb, 0);
            conv_tiles<prep::kThreads, prep::oV, 16384>(sm, a, n, h, hk, bos, t0, L, tid, gb, 1);
        }
    }
    if (ok && L < kC) {  // rows past the end of the sequence hold other tokens: zero them
        for (int e = tid; e < (kC - L) * 8 * 4; e += kThreads) {
            const int r = L + e / 32, part = e % 32;  // 4 tiles (K, Q x 2 halves) x 8 chunks of 16 B
            const int tile = part / 8, ch = part % 8;
            *reinterpret_cast<uint4*>(sm + oKQ + (tile & 1) * 16384 + (tile >> 1) * 8192 + r * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    if (ok && (a.conv.w || L < kC)) fence_async_smem();  // generic writes, read next by the MMA
    gb.sync();
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
            if (tid < kC) {
                const float diag = pick64(r0, r1, tid);  // k_i . k_i
                kinv[tid] = a.use_l2 ? rsqrtf(diag + kL2Eps) : 1.0f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) { row[j] = __uint_as_float(r0[j]); row[32 + j] = __uint_as_float(r1[j]); }
        }
        if (tid >= kC) {
            uint32_t r2[32], r3[32];
            tmem_ld32(lane_addr + 64, r2);
            tmem_ld32(lane_addr + 96, r3);
            tmem_wait_ld();
            const float diag = pick64(r2, r3, tid - kC);  // q_i . q_i
            qsv[tid - kC] = a.scale * (a.use_l2 ? rsqrtf(diag + kL2Eps) : 1.0f);
        }
        tc_fence_before();
        gb.sync();
        pc_products(sm, a, gh, h, t0, L, tid, kinv, qsv, bts, Af, Tf, gb);
        fence_async_smem();  // the K tile may have been rewritten (K . e^G) for the W product
        gb.sync();
        // Q is no longer read: V comes into its rows while the triangular solve runs
        if (tid == 0) {
            fence_async_smem();
            mbar_arrive_expect_tx(&bars[2], 16384);
            for (int c = 0; c < 2; ++c) tma_load_3d(sm + oV + c * 16384, mV, &bars[2], c * 64, h, (int)t0);
        }
        // ---- T = (I + A)^-1 ----
        unit_lower_inverse(Af, Tf, tid, gb);
        // ---- T' = T diag(beta e^gc kinv) and T'' = T diag(beta) as bf16 SW128 operand tiles ----
        if (tid < kC) qsv[tid] = bts[tid] * __expf(gcs[tid]) * kinv[tid];  // q factors no longer needed
        gb.sync();
        {
            const int i = tid & 63, which = tid >> 6;
            uint8_t* dst = sm + (which ? oTPP : oTP);
            const float* cfv = which ? bts : qsv;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = Tf[i * LD + c8 * 8 + e] * cfv[c8 * 8 + e];
                st_sw128_chunk(dst, i, c8, v);
            }
        }
        // V: landed, convolved, rows past the sequence zeroed
        const bool okv = mbar_wait(&bars[2], tma_parity, kPolls);
        if (a.conv.w && !gb.sync_or(!okv)) conv_tiles<prep::kThreads, prep::oV, 16384>(sm, a, n, h, hk, bos, t0, L, tid, gb, 2);
        if (okv && L < kC) {
            for (int e = tid; e < (kC - L) * 8 * 2; e += kThreads) {
                const int r = L + e / 16, part = e % 16;
                *reinterpret_cast<uint4*>(sm + oV + (part >> 3) * 16384 + r * 128 + (part & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        fence_async_smem();
        tc_fence_before();
        const bool vfail = gb.sync_or(!okv);
        if (vfail) {
            if (tid == 0) record_error(a.err, GDN_ERR_TIMEOUT);
        } else if (tid == 0) {
            tc_fence_after();
            const uint32_t kq = smem_u32(sm + oKQ), vv = smem_u32(sm + oV);
            const uint32_t tp = smem_u32(sm + oTP), tpp = smem_u32(sm + oTPP);
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tm + 0, sdesc_sw128(kq + k * 2048, 16384, 1024), sdesc_sw128(tp + k * 32, 16, 1024),
                            idesc_bf16(128, 64, 1, 0), k > 0);
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tm + 64, sdesc_sw128(vv + k * 2048, 16384, 1024), sdesc_sw128(tpp + k * 32, 16, 1024),
                            idesc_bf16(128, 64, 1, 0), k > 0);
            mma_commit(&bars[1]);
        }
        const bool ok2 = !vfail && mbar_wait(&bars[1], 1, kPolls);
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
                // U^T row tid (128 B), staged in the T tile (free once T' and T'' are built)
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(Tf) + tid * 128);
                const int sw = tid & 7;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    dst[c8 ^ sw] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c8]), __uint_as_float(r0[8 * c8 + 1])),
                                              pack_bf16x2(__uint_as_float(r0[8 * c8 + 2]), __uint_as_float(r0[8 * c8 + 3])),
                                              pack_bf16x2(__uint_as_float(r0[8 * c8 + 4]), __uint_as_float(r0[8 * c8 + 5])),
                                              pack_bf16x2(__uint_as_float(r0[8 * c8 + 6]), __uint_as_float(r0[8 * c8 + 7])));
                    dst[(4 + c8) ^ sw] = make_uint4(pack_bf16x2(__uint_as_float(r1[8 * c8]), __uint_as_float(r1[8 * c8 + 1])),
                                                    pack_bf16x2(__uint_as_float(r1[8 * c8 + 2]), __uint_as_float(r1[8 * c8 + 3])),
                                                    pack_bf16x2(__uint_as_float(r1[8 * c8 + 4]), __uint_as_float(r1[8 * c8 + 5])),
                                                    pack_bf16x2(__uint_as_float(r1[8 * c8 + 6]), __uint_as_float(r1[8 * c8 + 7])));
                }
            }
            gb.sync();
            const uint4* src = reinterpret_cast<const uint4*>(Wst);
            uint4* dst = reinterpret_cast<uint4*>(a.W + gh * kC * kD);
            for (int e = tid; e < kC * kD / 8; e += kThreads) dst[e] = src[e];
            const uint4* usrc = reinterpret_cast<const uint4*>(Tf);
            uint4* udst = reinterpret_cast<uint4*>(a.Ut + gh * kD * kC);
#pragma unroll
            for (int it = 0; it < 8; ++it) {  // 128 rows x 8 chunks; a warp writes 4 whole rows
                const int e = it * kThreads + tid, r = e >> 3;
                udst[e] = usrc[(r << 3) + ((e & 7) ^ (r & 7))];
            }
        }
    }
}

template <bool PC>
__global__ void __launch_bounds__(prep::kThreads, 3)
chunk_prep_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, TcArgs a) {
    using namespace prep;
    extern __shared__ uint8_t smraw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so that the compiler
    // keeps the shared address space (plain shared loads and stores, not generic ones)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oBar + 32);
    const int tid = threadIdx.x, warp = tid >> 5;
    const long gh = blockIdx.x;  // chunk * H + head
    if (gh / a.H >= a.n_chunks[0]) return;
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tmap(&mQ);
        prefetch_tmap(&mK);
        prefetch_tmap(&mV);
    }
    if (warp == 0) {
        tmem_alloc(tbase, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    prep_chunk<PC>(sm, tm, bars, 0, GroupBar{1}, tid, gh, &mQ, &mK, &mV, a);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// ---- 2b. chunk preparation by eight warps (decay per head) -------------------------------------
//
// The same entries as prep_chunk, computed by 256 threads so that every phase's work per thread
// halves and two chunks in flight keep 16 warps busy on an SM:
//  - the K, Q and V tiles are requested together as the chunk starts;
//  - the norms are summed from the loaded tiles while the Gram product [K; Q] K^T runs (N = 64:
//    only the key columns of the Gram matrix are used);
//  - the decays enter in the log domain: A_ij = 2^(cA_i - dK_j) (K K^T)_ij with
//    cA_i = gc_i log2(e) + log2(beta_i kinv_i) and dK_j = gc_j log2(e) - log2(kinv_j), and
//    Aqk_ij = 2^(cQ_i - dK_j) (Q K^T)_ij with cQ_i = gc_i log2(e) + log2(qs_i): one exponential and
//    one product per element.  Where an element is kept (j < i, or j <= i) gc_i <= gc_j, so the
//    exponent is at most log2 of the norm factors and nothing overflows;
//  - T = (I + A)^-1 by block doubling.  Warps 0 and 1 each invert two 16 x 16 diagonal blocks by
//    forward substitution and merge them, T_10 = -t_11 A_10 t_00 and T_32 = -t_33 A_32 t_22,
//    synchronising only within the warp, while warps 2-7 write the state pass's scaled operand
//    rows; then all eight warps take the 64 x 64 merge T_hl = -T_hh A_hl T_ll in 8 x 16 pieces.
//    Every piece of T is written at once in fp32 (for the later merges) and as bf16 entries of the
//    operand tiles T' = T diag(beta e^gc kinv) and T'' = T diag(beta), whose upper triangles are
//    zeroed once per CTA and never written;
//  - Aqk, W and U^T are staged in shared memory and leave in whole 512-byte rows per warp.
namespace p2 {
constexpr int kThreads = 256;
constexpr int LDA = kC + 1;                    // A (fp32 64 x 64), odd row stride
constexpr int LD = kC + 4;                     // T (fp32 64 x 64); its rows 0-31, columns 32-63 lie
                                               // above the diagonal and serve the solve as scratch
constexpr uint32_t oKQ = 0;                    // K rows 0-63 and Q rows 64-127 in two atom columns
constexpr uint32_t oV = 32768;                 // V: two atom columns of 64 rows, 8 KB apart
constexpr uint32_t oAf = 49152;                // A; after the products the W staging (64 x 256 B)
constexpr uint32_t oTf = oAf + 16896;          // T; after the products the U^T staging (128 x 128 B)
constexpr uint32_t oTP = 83968;                // T' and T'' (bf16 SW128 64 x 64, 8 KB each)
constexpr uint32_t oAqk = oTP + 16384;         // Aqk staging (64 x 128 B, 16-byte pieces swizzled)
constexpr uint32_t oSc = oAqk + 8192;          // per-token scalars: 10 rows of 64 fp32
constexpr uint32_t oBar = oSc + 10 * 4 * kC;   // mbarriers (K and Q, products, V), then the TMEM base
constexpr uint32_t kBytes = oBar + 64;
constexpr uint32_t kSmem = kBytes + 1024;      // + alignment slack
constexpr uint32_t kTmemCols = 128;            // the Gram product (64 columns), then W^T and U^T
static_assert(oTf + 4 * kC * LD <= oTP && (oTP & 1023u) == 0, "layout");
static_assert(2 * (kSmem + 1024) <= 233472, "two chunks per SM");
enum { S_GC = 0, S_BETA, S_KINV, S_QS, S_CA, S_CQ, S_DK, S_KF, S_QF, S_TP };  // scalar rows
}  // namespace p2

// C[8 x 16] (+)= P[8 x 16] Q[16 x 16] for one warp: lane l owns row l / 4 and columns
// 4 (l % 4) .. 4 (l % 4) + 3 of C.  P and Q are fp32 in shared memory with row strides LDP and LDQ
// (LDQ a multiple of 4).
template <int LDP, int LDQ>
__device__ __forceinline__ void warp_mm8(const float* P, const float* Q, float (&c)[4], int lane) {
    const int ii = lane >> 2, c0 = (lane & 3) * 4;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float p = P[ii * LDP + k];
        const float4 q = *reinterpret_cast<const float4*>(Q + k * LDQ + c0);
        c[0] = fmaf(p, q.x, c[0]); c[1] = fmaf(p, q.y, c[1]); c[2] = fmaf(p, q.z, c[2]); c[3] = fmaf(p, q.w, c[3]);
    }
}

// Row `row`, columns col .. col + 3 of T (fp32, negated when `neg`) into T and, scaled, into the
// bf16 operand tiles T' and T''.
__device__ __forceinline__ void put_t4(uint8_t* sm, float* Tf, const float* sc, int row, int col, const float (&c)[4],
                                       bool neg) {
    using namespace p2;
    const float4 t = neg ? make_float4(-c[0], -c[1], -c[2], -c[3]) : make_float4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<float4*>(Tf + row * LD + col) = t;
    const float4 f = *reinterpret_cast<const float4*>(sc + S_TP * kC + col);
    const float4 b = *reinterpret_cast<const float4*>(sc + S_BETA * kC + col);
    const uint32_t off = sw128_offset(row, col);
    *reinterpret_cast<uint2*>(sm + oTP + off) = make_uint2(pack_bf16x2(t.x * f.x, t.y * f.y), pack_bf16x2(t.z * f.z, t.w * f.w));
    *reinterpret_cast<uint2*>(sm + oTP + 8192 + off) =
        make_uint2(pack_bf16x2(t.x * b.x, t.y * b.y), pack_bf16x2(t.z * b.z, t.w * b.w));
}

// Inverse of the unit lower-triangular 16 x 16 diagonal block at (b0, b0) of I + A by forward
// substitution; lane jj (0..15) computes column jj (entries above the diagonal come out zero) and
// writes it to T, T' and T''.
__device__ __forceinline__ void diag_inverse16(uint8_t* sm, const float* Af, float* Tf, const float* sc, int b0, int jj) {
    using namespace p2;
    float t[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
        // t[m] is zero for m < jj, so the sum may run over every m < ii
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int m = 0; m < ii; ++m) {
            if (m & 1) acc1 = fmaf(Af[(b0 + ii) * LDA + b0 + m], t[m], acc1);
            else acc0 = fmaf(Af[(b0 + ii) * LDA + b0 + m], t[m], acc0);
        }
        t[ii] = ii < jj ? 0.f : (ii == jj ? 1.f : -(acc0 + acc1));
    }
    const int j = b0 + jj;
    const float fj = sc[S_TP * kC + j], bj = sc[S_BETA * kC + j];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
        Tf[(b0 + ii) * LD + j] = t[ii];
        const uint32_t off = sw128_offset(b0 + ii, j);
        *reinterpret_cast<__nv_bfloat16*>(sm + oTP + off) = __float2bfloat16_rn(t[ii] * fj);
        *reinterpret_cast<__nv_bfloat16*>(sm + oTP + 8192 + off) = __float2bfloat16_rn(t[ii] * bj);
    }
}

// Zero the operand tiles T' and T'' (their upper triangles are never written afterwards); run by
// every thread of a preparation group before its first chunk.
__device__ __forceinline__ void prep2_init_tiles(uint8_t* sm, int tid) {
    for (int e = tid; e < 16384 / 16; e += p2::kThreads)
        reinterpret_cast<uint4*>(sm + p2::oTP)[e] = make_uint4(0, 0, 0, 0);
}

// Where chunk-head item gh = chunk * H + head lies in the packed tokens.
struct ChunkPos {
    long gh, t0, bos;
    int n, h, hk, L;
};
__device__ __forceinline__ ChunkPos chunk_pos(const TcArgs& a, long gh) {
    ChunkPos p;
    p.gh = gh;
    const int chunk = (int)(gh / a.H);
    p.h = (int)(gh % a.H);
    p.hk = p.h / (a.H / a.Hk);  // query/key head read by value head h
    p.n = a.chunk_seq[chunk];
    long eos;
    seq_bounds(a, p.n, p.bos, eos);
    p.t0 = p.bos + (long)(chunk - a.chunk_first[p.n]) * kC;
    p.L = (eos - p.t0 < kC) ? (int)(eos - p.t0) : kC;
    return p;
}

// Thread 0: request the K, Q (one barrier) and V (another) tiles of chunk p.
__device__ __forceinline__ void prep2_issue(uint8_t* sm, uint64_t* bars, const ChunkPos& p, const CUtensorMap* mQ,
                                            const CUtensorMap* mK, const CUtensorMap* mV) {
    using namespace p2;
    fence_async_smem();  // earlier generic accesses to the tiles come first
    mbar_arrive_expect_tx(&bars[0], 32768);
    for (int c = 0; c < 2; ++c) {
        tma_load_3d(sm + oKQ + c * 16384, mK, &bars[0], c * 64, p.hk, (int)p.t0);
        tma_load_3d(sm + oKQ + c * 16384 + 8192, mQ, &bars[0], c * 64, p.hk, (int)p.t0);
    }
    mbar_arrive_expect_tx(&bars[2], 16384);
    for (int c = 0; c < 2; ++c) tma_load_3d(sm + oV + c * 8192, mV, &bars[2], c * 64, p.h, (int)p.t0);
}

// Warp 0: g, warp 1: beta of tokens 2 lane and 2 lane + 1 of chunk p into x0, x1 (zero past the
// sequence).  Other warps leave x0, x1 alone.  Only loads: the values are first used at the start
// of the chunk, so a prefetch leaves them in flight meanwhile.
__device__ __forceinline__ void prep2_load_gb(const TcArgs& a, const ChunkPos& p, int warp, int lane, float& x0, float& x1) {
    const int i0 = 2 * lane;
    if (warp < 2) {
        const float* src = (warp == 0 ? a.g : a.beta) + p.t0 * a.H + p.h;
        x0 = i0 < p.L ? src[(long)i0 * a.H] : 0.f;
        x1 = i0 + 1 < p.L ? src[(long)(i0 + 1) * a.H] : 0.f;
    }
}

// One chunk of one head by 256 threads (tid 0..255, synchronised by `gb`): everything the state
// pass needs from it, written to the workspace.  `sm` is the chunk's 1024-aligned shared region,
// `tm` its 128 TMEM columns, `bars` its three mbarriers; the tile barriers complete with parity
// `tma_parity`.  When `loaded`, the chunk's tiles were requested and its g / beta values (x0, x1
// of warps 0 and 1, see prep2_load_gb) loaded during the previous chunk.  With `more`, the next
// chunk `nxt`'s tiles are requested as soon as this chunk's products have read the tiles, and its
// g / beta go to x0, x1.  Returns false after a timed-out wait (recorded in the error word);
// the tile copies in flight have then landed or timed out too.
__device__ __forceinline__ bool prep2_chunk(uint8_t* sm, uint32_t tm, uint64_t* bars, uint32_t tma_parity,
                                            GroupBar gb, int tid, const ChunkPos& cur, bool loaded,
                                            const ChunkPos& nxt, bool more, float& x0, float& x1, const CUtensorMap* mQ,
                                            const CUtensorMap* mK, const CUtensorMap* mV, const TcArgs& a) {
    using namespace p2;
    constexpr float kLog2e = 1.4426950408889634f;
    float* Af = reinterpret_cast<float*>(sm + oAf);
    float* Tf = reinterpret_cast<float*>(sm + oTf);
    float* sc = reinterpret_cast<float*>(sm + oSc);
    const int warp = tid >> 5, lane = tid & 31;
    const long gh = cur.gh, t0 = cur.t0, bos = cur.bos;
    const int n = cur.n, h = cur.h, hk = cur.hk, L = cur.L;
    auto fail = [&]() {
        if (tid == 0) {
            record_error(a.err, GDN_ERR_TIMEOUT);
            mbar_wait(&bars[0], tma_parity, kPolls);  // no tile copy may still be in flight
            mbar_wait(&bars[2], tma_parity, kPolls);
        }
        return false;
    };

    if (!loaded) {
        if (tid == 0) prep2_issue(sm, bars, cur, mQ, mK, mV);
        prep2_load_gb(a, cur, warp, lane, x0, x1);
    }
    if (warp == 0) {  // gc: inclusive sums of g down the chunk, two tokens per lane
        float sum = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, sum, o);
            if (lane >= o) sum += t;
        }
        sc[S_GC * kC + 2 * lane] = sum - x1;
        sc[S_GC * kC + 2 * lane + 1] = sum;
    } else if (warp == 1) {
        sc[S_BETA * kC + 2 * lane] = x0;
        sc[S_BETA * kC + 2 * lane + 1] = x1;
    }
    const bool ok = mbar_wait(&bars[0], tma_parity, kPolls);
    if (gb.sync_or(!ok)) return fail();
    if (a.conv.w) {  // fused short convolution of the loaded rows
        conv_tiles<kThreads, oV, 8192>(sm, a, n, h, hk, bos, t0, L, tid, gb, 0);
        conv_tiles<kThreads, oV, 8192>(sm, a, n, h, hk, bos, t0, L, tid, gb, 1);
    }
    if (L < kC) {  // rows past the end of the sequence hold other tokens: zero them
        for (int e = tid; e < (kC - L) * 8 * 4; e += kThreads) {
            const int r = L + e / 32, part = e % 32;  // 4 tiles (K, Q x 2 atom columns) x 8 pieces of 16 B
            const int tile = part / 8, ch = part % 8;
            *reinterpret_cast<uint4*>(sm + oKQ + (tile & 1) * 16384 + (tile >> 1) * 8192 + r * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    if (a.conv.w || L < kC) fence_async_smem();  // generic writes to the tiles, read next by the tensor cores
    gb.sync();
    if (tid == 0) {  // Gram product: rows [K; Q] (M = 128) against the key rows (N = 64)
        tc_fence_after();
        const uint32_t kq = smem_u32(sm + oKQ);
        for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_bf16_ss(tm, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024),
                        idesc_bf16(128, 64, 0, 0), k > 0);
        }
        mma_commit(&bars[1]);
    }
    {   // norms from the tiles: a quarter-warp takes 8 rows (8 distinct swizzle phases) of one atom
        // column, the partner lane (lane ^ 8) the other column of the same rows
        const int r = warp * 16 + (lane & 7) + ((lane >> 4) << 3);  // K rows 0-63, then Q rows
        const int hc = (lane >> 3) & 1;
        const uint8_t* rowp = sm + oKQ + hc * 16384 + (r >> 6) * 8192 + (r & 63) * 128;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float f[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rowp + ((c ^ (r & 7)) << 4)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) s4[e & 3] = fmaf(f[e], f[e], s4[e & 3]);
        }
        float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        if (hc == 0) {
            const float inv = a.use_l2 ? rsqrtf(ss + kL2Eps) : 1.0f;
            if (r < kC) sc[S_KINV * kC + r] = inv;
            else sc[S_QS * kC + r - kC] = a.scale * inv;
        }
    }
    gb.sync();
    if (tid < kC) {  // per-token factors
        const int i = tid;
        const float gi = sc[S_GC * kC + i], glast = sc[S_GC * kC + kC - 1];
        const float bt = sc[S_BETA * kC + i], ki = sc[S_KINV * kC + i], qs = sc[S_QS * kC + i];
        const float egi = __expf(gi);
        sc[S_CA * kC + i] = gi * kLog2e + __log2f(bt * ki);
        sc[S_CQ * kC + i] = gi * kLog2e + __log2f(qs);
        sc[S_DK * kC + i] = gi * kLog2e - __log2f(ki);
        sc[S_KF * kC + i] = __expf(glast - gi) * ki;   // K~ rows
        sc[S_QF * kC + i] = egi * qs;                  // Q~ rows
        sc[S_TP * kC + i] = bt * egi * ki;             // columns of T' = T diag(beta e^gc kinv)
        if (i == 0) a.scal[gh * 4 * kC + 3 * kC] = __expf(glast);  // the chunk's decay gamma
    }
    const bool okg = mbar_wait(&bars[1], 0, kPolls);
    tc_fence_after();
    if (gb.sync_or(!okg)) return fail();
    {   // ---- E1: Gram rows -> A (fp32, shared) and Aqk (bf16, staged) ----
        // warp: TMEM lanes 32 q4 .. 32 q4 + 31 (Gram rows: K rows for q4 < 2, Q rows above),
        // columns j0 .. j0 + 31
        const int q4 = warp & 3, j0 = 32 * (warp >> 2);
        const bool isq = q4 >= 2;
        const int i = 32 * (q4 & 1) + lane;              // token of the row
        const int lim = isq ? i + 1 : i;                 // kept columns: j < lim
        const bool empty = j0 == 32 && (q4 & 1) == 0;    // every column of the warp lies past its rows
        uint4* stage = reinterpret_cast<uint4*>(sm + oAqk + i * 128);  // Aqk row i: piece c at c ^ (i & 7)
        if (!empty) {
            uint32_t r[32];
            tmem_ld32(tm + (static_cast<uint32_t>(32 * q4) << 16) + (uint32_t)j0, r);
            tmem_wait_ld();
            const float ci = sc[(isq ? S_CQ : S_CA) * kC + i];
            const float* dk = sc + S_DK * kC + j0;
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float x = ex2_approx(ci - dk[e]) * __uint_as_float(r[e]);
                v[e] = j0 + e < lim ? x : 0.f;
            }
            if (!isq) {
#pragma unroll
                for (int e = 0; e < 32; ++e) Af[i * LDA + j0 + e] = v[e];
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) stage[((j0 >> 3) + c) ^ (i & 7)] = pack_bf16x8(v + 8 * c);
            }
        } else if (isq) {
#pragma unroll
            for (int c = 0; c < 4; ++c) stage[((j0 >> 3) + c) ^ (i & 7)] = make_uint4(0, 0, 0, 0);
        }
    }
    tc_fence_before();
    gb.sync();
    if (warp < 2) {
        // ---- warp w: diagonal blocks 2w (lanes 0-15) and 2w + 1 (lanes 16-31), then their merge
        //      T_{b,b-1} = -t_b (A_{b,b-1} t_{b-1}), b = 2w + 1 ----
        diag_inverse16(sm, Af, Tf, sc, 32 * warp + 16 * (lane >> 4), lane & 15);
        __syncwarp();
        const int b = 2 * warp + 1;
        float* Y = Tf + 32 + 16 * warp;  // scratch: rows 0-15 of T, columns 32 + 16 w ..
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
            warp_mm8<LDA, LD>(Af + (16 * b + 8 * hh) * LDA + 16 * (b - 1), Tf + 16 * (b - 1) * LD + 16 * (b - 1), c[hh], lane);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
            *reinterpret_cast<float4*>(Y + (8 * hh + (lane >> 2)) * LD + (lane & 3) * 4) =
                make_float4(c[hh][0], c[hh][1], c[hh][2], c[hh][3]);
        __syncwarp();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            warp_mm8<LD, LD>(Tf + (16 * b + 8 * hh) * LD + 16 * b, Y, d, lane);
            put_t4(sm, Tf, sc, 16 * b + 8 * hh + (lane >> 2), 16 * (b - 1) + (lane & 3) * 4, d, true);
        }
    } else {
        // ---- meanwhile: the operand rows K~ = diag(kf) K and Q~ = diag(qf) Q (2 tensors x 64 rows
        //      x 16 pieces of 16 B over 192 threads; a warp writes 2 whole rows), then Aqk ----
#pragma unroll
        for (int it = 0; it < 11; ++it) {
            const int flat = it * (kThreads - 64) + tid - 64;
            if (flat < 2048) {
                const int isq = flat >> 10, r = (flat >> 4) & 63, c16 = flat & 15;
                const uint4 raw = *reinterpret_cast<const uint4*>(sm + oKQ + (c16 >> 3) * 16384 + (isq ? 8192 : 0) +
                                                                  sw128_offset(r, (c16 & 7) * 8));
                const float fr = sc[(isq ? S_QF : S_KF) * kC + r];
                float v[8];
                unpack_bf16x8(raw, v);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] *= fr;
                *reinterpret_cast<uint4*>((isq ? a.Qt : a.Kt) + gh * kC * kD + (long)r * kD + c16 * 8) = pack_bf16x8(v);
            }
        }
        uint4* adst = reinterpret_cast<uint4*>(a.Aqk + gh * kC * kC);
#pragma unroll
        for (int it = 0; it < 3; ++it) {  // 64 rows x 8 pieces
            const int flat = it * (kThreads - 64) + tid - 64;
            if (flat < 512) {
                const int r = flat >> 3, c8 = flat & 7;
                adst[flat] = reinterpret_cast<const uint4*>(sm + oAqk + r * 128)[c8 ^ (r & 7)];
            }
        }
    }
    gb.sync();
    {   // ---- the 64 x 64 merge: X = A_hl T_ll, then T_hl = -T_hh X, as 2 x 2 blocks of 16 ----
        // warp: output block (p, q) of the 32 x 32 result, rows r8 .. r8 + 7 of it
        float* X = Tf + 32;  // scratch: rows 0-31, columns 32-63 of T
        const int p = warp >> 2, q = (warp >> 1) & 1, r8 = (warp & 1) * 8;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = q; k < 2; ++k)  // T_ll is lower triangular: block (k, q) vanishes for k < q
            warp_mm8<LDA, LD>(Af + (32 + 16 * p + r8) * LDA + 16 * k, Tf + 16 * k * LD + 16 * q, c, lane);
        *reinterpret_cast<float4*>(X + (16 * p + r8 + (lane >> 2)) * LD + 16 * q + (lane & 3) * 4) =
            make_float4(c[0], c[1], c[2], c[3]);
        gb.sync();
        c[0] = c[1] = c[2] = c[3] = 0.f;
        for (int k = 0; k <= p; ++k)  // T_hh is lower triangular: block (p, k) vanishes for k > p
            warp_mm8<LD, LD>(Tf + (32 + 16 * p + r8) * LD + 32 + 16 * k, X + 16 * k * LD + 16 * q, c, lane);
        put_t4(sm, Tf, sc, 32 + 16 * p + r8 + (lane >> 2), 16 * q + (lane & 3) * 4, c, true);
    }
    // V: landed, convolved, rows past the sequence zeroed
    const bool okv = mbar_wait(&bars[2], tma_parity, kPolls);
    if (gb.sync_or(!okv)) return fail();
    if (a.conv.w) conv_tiles<kThreads, oV, 8192>(sm, a, n, h, hk, bos, t0, L, tid, gb, 2);
    if (L < kC) {
        for (int e = tid; e < (kC - L) * 16; e += kThreads) {
            const int r = L + e / 16, part = e % 16;
            *reinterpret_cast<uint4*>(sm + oV + (part >> 3) * 8192 + r * 128 + (part & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_async_smem();  // T', T'' and any rewritten V rows, read next by the tensor cores
    gb.sync();
    if (tid == 0) {  // W^T = K^T T'^T and U^T = V^T T''^T (K and V as MN-major operands)
        tc_fence_after();
        const uint32_t kq = smem_u32(sm + oKQ), vv = smem_u32(sm + oV);
        const uint32_t tp = smem_u32(sm + oTP), tpp = tp + 8192;
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
    if (gb.sync_or(!ok2)) return fail();
    if (more) {  // the products have read the tiles: the next chunk's tiles and scalars now
        if (tid == 0) prep2_issue(sm, bars, nxt, mQ, mK, mV);
        prep2_load_gb(a, nxt, warp, lane, x0, x1);
    }
    {   // ---- E2: W (token-major) and U^T (row per value channel), staged over A and T ----
        // thread: TMEM lane d = key channel (W^T) and value channel (U^T), tokens 32 th .. 32 th + 31
        const int q4 = warp & 3, th = warp >> 2;
        const int d = 32 * q4 + lane;
        const uint32_t lrow = static_cast<uint32_t>(32 * q4) << 16;
        uint32_t w[32], u[32];
        tmem_ld32(tm + lrow + (uint32_t)(32 * th), w);
        tmem_ld32(tm + lrow + 64u + (uint32_t)(32 * th), u);
        tmem_wait_ld();
        __nv_bfloat16* wst = reinterpret_cast<__nv_bfloat16*>(sm + oAf) + (32 * th) * kD + d;  // [64][128]
#pragma unroll
        for (int e = 0; e < 32; ++e) wst[e * kD] = __float2bfloat16_rn(__uint_as_float(w[e]));
        uint4* ust = reinterpret_cast<uint4*>(sm + oTf + d * 128);  // U^T row d: piece c at c ^ (d & 7)
#pragma unroll
        for (int c = 0; c < 4; ++c) ust[(4 * th + c) ^ (d & 7)] = pack_bf16x8(reinterpret_cast<const float*>(u) + 8 * c);
    }
    tc_fence_before();
    gb.sync();
    {   // whole rows out: W 1024 pieces of 16 B, U^T 1024
        uint4* wdst = reinterpret_cast<uint4*>(a.W + gh * kC * kD);
        uint4* udst = reinterpret_cast<uint4*>(a.Ut + gh * kD * kC);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = it * kThreads + tid;
            wdst[e] = reinterpret_cast<const uint4*>(sm + oAf)[e];
            const int r = e >> 3;
            udst[e] = reinterpret_cast<const uint4*>(sm + oTf + r * 128)[(e & 7) ^ (r & 7)];
        }
    }
    gb.sync();  // every read of this chunk's tiles, scalars and TMEM is done
    return true;
}

__global__ void __launch_bounds__(p2::kThreads, 2)
chunk_prep2_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mV, TcArgs a) {
    using namespace p2;
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oBar + 32);
    const int tid = threadIdx.x, warp = tid >> 5;
    const long n_items = (long)a.n_chunks[0] * a.H;  // chunk-head pairs, item gh = chunk * H + head
    if ((long)blockIdx.x >= n_items) return;
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tmap(&mQ);
        prefetch_tmap(&mK);
        prefetch_tmap(&mV);
    }
    if (warp == 0) {
        tmem_alloc(tbase, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    prep2_init_tiles(sm, tid);
    uint32_t parity = 0;
    float x0 = 0.f, x1 = 0.f;
    ChunkPos cur = chunk_pos(a, blockIdx.x);
    bool loaded = false;
    for (long gh = blockIdx.x; gh < n_items; gh += gridDim.x) {
        const bool more = gh + gridDim.x < n_items;
        const ChunkPos nxt = more ? chunk_pos(a, gh + gridDim.x) : cur;
        if (!prep2_chunk(sm, tm, bars, parity, GroupBar{1, kThreads}, tid, cur, loaded, nxt, more, x0, x1, &mQ, &mK,
                         &mV, a))
            break;
        parity ^= 1u;
        cur = nxt;
        loaded = more;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// 64 columns of this thread's two rows of an M = 64 accumulator (16x256b shape, 16 repetitions)
__device__ __forceinline__ void tmem_ld16x256b_x16(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
          "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
          "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
          "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
          "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
        : "r"(taddr));
}

// ---- the gated output of one chunk, shared by the serial pass and the output items ----------------
//
// O (M = 64, tokens as rows) comes out of TMEM with a 16x256b load: this thread holds rows
// rA = 16 q + lane / 4 and rA + 8 and, in every group of 8 columns, the pair cp, cp + 1
// (cp = 2 (lane % 4)); o[4 j + {0,1}] belong to row rA, o[4 j + {2,3}] to row rA + 8.

// Each row's sum of squares over d_v: the four lanes of a row add their shares with two shuffles.
__device__ __forceinline__ void out_sumsq(const float* o, float& ssA, float& ssB) {
    float sA0 = 0.f, sA1 = 0.f, sB0 = 0.f, sB1 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        sA0 = fmaf(o[4 * j], o[4 * j], sA0);
        sA1 = fmaf(o[4 * j + 1], o[4 * j + 1], sA1);
        sB0 = fmaf(o[4 * j + 2], o[4 * j + 2], sB0);
        sB1 = fmaf(o[4 * j + 3], o[4 * j + 3], sB1);
    }
    ssA = sA0 + sA1;
    ssB = sB0 + sB1;
    ssA += __shfl_xor_sync(0xffffffffu, ssA, 1);
    ssB += __shfl_xor_sync(0xffffffffu, ssB, 1);
    ssA += __shfl_xor_sync(0xffffffffu, ssA, 2);
    ssB += __shfl_xor_sync(0xffffffffu, ssB, 2);
}

// The RMS norm and SiLU gate (when a.z is set; z of the chunk in the 128-byte-swizzled tile zt, four
// boxes of [64 tokens][32 fp32]) and the stores of the chunk's rows t0 .. t0 + L - 1, by the 128
// threads of named barrier gbar.  A full chunk with bf16 output is staged in zt as two [64 x 64]
// boxes (after every row has read its z) and stored by the leader with the output's tensor map (the
// caller commits nothing further and waits for the store before reusing zt); otherwise the rows
// inside the sequence are written directly.  Nothing is stored unless ok.
__device__ __forceinline__ void out_gate_store(float* o, float ssA, float ssB, int rA, int cp, uint8_t* zt, bool ok,
                                               int L, long t0, int h, bool leader, uint32_t gbar,
                                               const CUtensorMap* mOut, const TcArgs& a) {
    const long tok_stride = (long)a.H * a.d;
    const bool bf16_out = a.out_dtype == GDN_BF16;
    if (a.z) {
        // the mean over the head's d_v outputs (the padded columns are zeros)
        const float rA_inv = rsqrtf(ssA / a.d + a.eps), rB_inv = rsqrtf(ssB / a.d + a.eps);
        // bf16 output: SiLU with the packed half-precision tanh (error near 1e-3, below the
        // output's 2^-9 rounding); fp32 output: SiLU at fp32 accuracy.  The choice is taken once,
        // outside the loop, so that only one of the two is evaluated per element.
        auto gate = [&](auto silu2) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int col = 8 * j + cp, cb = col >> 5, ch = (col & 31) >> 2, sub = (col & 3) * 4;
                const float2 zA = *reinterpret_cast<const float2*>(zt + cb * 8192 + rA * 128 + ((ch ^ (rA & 7)) << 4) + sub);
                const float2 zB = *reinterpret_cast<const float2*>(zt + cb * 8192 + (rA + 8) * 128 +
                                                                   ((ch ^ ((rA + 8) & 7)) << 4) + sub);
                float2 wA = make_float2(rA_inv, rA_inv), wB = make_float2(rB_inv, rB_inv);
                if (a.w && col < a.d) {
                    const float2 wv = __ldg(reinterpret_cast<const float2*>(a.w + col));
                    wA = make_float2(wv.x * rA_inv, wv.y * rA_inv);
                    wB = make_float2(wv.x * rB_inv, wv.y * rB_inv);
                }
                const float2 sA = silu2(zA), sB = silu2(zB);
                o[4 * j] *= wA.x * sA.x;
                o[4 * j + 1] *= wA.y * sA.y;
                o[4 * j + 2] *= wB.x * sB.x;
                o[4 * j + 3] *= wB.y * sB.y;
            }
        };
        if (bf16_out)
            gate([](float2 x) { return fast_silu2(x.x, x.y); });
        else
            gate([](float2 x) { return make_float2(x.x * sigmoidf_(x.x), x.y * sigmoidf_(x.y)); });
    }
    if (bf16_out && L == kC) {
        // a full chunk: stage the bf16 rows as two 128-byte-swizzled [64 x 64] boxes in the chunk's
        // own z buffer (after every row has read its z) and let one thread store them with the
        // tensor map of the output
        if (a.z) bar_sync(gbar, 128);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            uint8_t* box = zt + (j >> 3) * 8192;
            const int cj = j & 7;
            *reinterpret_cast<uint32_t*>(box + rA * 128 + ((cj ^ (rA & 7)) << 4) + cp * 2) =
                pack_bf16x2(o[4 * j], o[4 * j + 1]);
            *reinterpret_cast<uint32_t*>(box + (rA + 8) * 128 + ((cj ^ ((rA + 8) & 7)) << 4) + cp * 2) =
                pack_bf16x2(o[4 * j + 2], o[4 * j + 3]);
        }
        fence_async_smem();
        bar_sync(gbar, 128);
        if (leader && ok) {
            tma_store_3d(mOut, zt, 0, h, (int)t0);
            if (a.d > 64) tma_store_3d(mOut, zt + 8192, 64, h, (int)t0);
            bulk_commit();
        }
    } else if (ok) {
        // a partial chunk (the last of its sequence) or an fp32 output: the rows inside the
        // sequence are written directly, two columns per store
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = rA + 8 * hr;
            if (r < L) {
                const long base = (t0 + r) * tok_stride + (long)h * a.d + cp;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (8 * j >= a.d) break;
                    const float x0 = o[4 * j + 2 * hr], x1 = o[4 * j + 2 * hr + 1];
                    if (bf16_out)
                        *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + base + 8 * j) =
                            pack_bf16x2(x0, x1);
                    else
                        *reinterpret_cast<float2*>(static_cast<float*>(a.out) + base + 8 * j) = make_float2(x0, x1);
                }
            }
        }
    }
}

// ---- 3. serial state pass ------------------------------------------------------------------------

namespace st {
constexpr int kThreads = 512;               // 16 warps = 4 warpgroups
// register split: launched at 128 per thread (512 x 128 = 65536); the producer / MMA warpgroup
// gives back down to 56, the state epilogue rises to 208 and the two output groups settle at 120:
// 128 x 56 + 128 x 208 + 256 x 120 = 64512
constexpr int kRegsLow = 56, kRegsHigh = 208, kRegsOut = 120;
static_assert(128 * kRegsLow + 128 * kRegsHigh + 256 * kRegsOut <= kThreads * 128, "register split");
constexpr uint32_t oS = 0;                  // S bf16 operand: 2 atom columns x 128 rows = 32 KB
constexpr uint32_t oA1 = 32768;             // V_new^T bf16 [128 x 64] SW128 = 16 KB
constexpr uint32_t oStage = 49152;          // two stages
// stage layout
constexpr uint32_t sWQ = 0;                 // 2 atom columns x (W rows 0-63, Q~ rows 64-127) = 32 KB
constexpr uint32_t sK = 32768;              // K~: 2 atom columns x 64 rows = 16 KB
constexpr uint32_t sAqk = 49152;            // 64 x 64 = 8 KB
constexpr uint32_t kStage = 57344;          // multiple of 1024
constexpr uint32_t oZ = oStage + 2 * kStage;     // gate input z, two buffers of 4 boxes of
                                                 // [64 tokens][32 fp32] SW128 = 2 x 32 KB
constexpr uint32_t oBar = oZ + 2 * 32768;
constexpr uint32_t oGam = oBar + 256;       // decay per key channel: next chunk's e^(gc_last), 2 x 128 fp32
constexpr uint32_t kBytes = oGam + 1024;
constexpr uint32_t kSmem = kBytes + 1024;
static_assert(kSmem <= 232448, "state kernel shared memory exceeds the per-block limit");
constexpr uint32_t kStageTx = 32768 + 16384 + 8192;
// barriers
enum { FULL0 = 0, FULL1, EMPTY0, EMPTY1, SBF, DA1, A12, SFULL, DO_0, DO_1, DOE_0, DOE_1, ZFULL0, ZFULL1, SCP, VCP, NBAR };
static_assert(8 * NBAR + 8 <= 256, "barrier block");
// export form: the stage holds W, K~ and U^T (two boxes of 64 rows where the combined form keeps Q~),
// and the chunk's decay gamma in a slot of the oGam row
constexpr uint32_t kStageTxExport = 16384 + 16384 + 16384;
constexpr uint32_t kTmemCols = 512;
}  // namespace st

// TMEM columns of the state CTA: S [0,128); S W^T (M=128, 64 columns) x 2 buffers [128,256);
// O = Q~ S^T + Aqk V_new (M=64, rows = tokens, 128 columns) x 2 buffers [256,512).
// The serial pass of one (sequence, head) unit by the whole CTA (512 threads).  When a.ready is set
// (fused kernel) the chunks' workspace entries are produced concurrently by other CTAs: the TMA
// producer and the state epilogue wait for a chunk's ready flag before they read its entries.  The
// epilogue's read-only-path loads (__ldg) of those entries stay correct there: every entry is
// first touched after its flag is acquired, each chunk's entries fill whole aligned slots (no
// cache line holds two chunks), and the SM runs no other CTA, so no stale line can be cached.
//
// With EXP (export form, fused kernel only, a.Sx set) the serial pass forms no output: per chunk it copies
// the state's operand tile and V_new^T to the workspace (warp 2, bulk copies) and flags them, and the
// output of the chunk is formed elsewhere (out_chunk).  The chain then waits, before rewriting either
// tile, for the copy to have read it (normally long done).
template <bool PC, bool EXP>
__device__ __forceinline__ void state_unit(uint8_t* sm, int unit, const CUtensorMap* mQt, const CUtensorMap* mKt,
                                           const CUtensorMap* mW, const CUtensorMap* mAqk,
                                           const CUtensorMap* mZ, const CUtensorMap* mOut, const CUtensorMap* mUt,
                                           const TcArgs& a) {
    using namespace st;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oBar + 8 * NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oBar + 8 * NBAR + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = unit / a.H, h = unit % a.H;
    long bos, eos;
    if (!seq_bounds(a, n, bos, eos)) return;  // reported by the chunk map kernel
    const int nck = (int)((eos - bos + kC - 1) / kC);
    const int first = a.chunk_first[n];
    constexpr bool exp = EXP;

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
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
    const uint32_t tS = tm, tDA0 = tm + 128, tDO0 = tm + 256;

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
                const long ghc = (long)(first + c) * a.H + h;
                if (a.ready) {
                    if (!wait_ready(a.ready + ghc)) { fail(); break; }
                    fence_proxy_async_global();  // the entries were written by generic stores
                }
                uint8_t* sp = stage_ptr(s);
                const int row = (int)(ghc * kC);
                // export form: gamma into its slot before the arrive that releases it with the stage
                if (exp) reinterpret_cast<float*>(sm + oGam)[s] = __ldg(a.scal + ghc * 4 * kC + 3 * kC);
                mbar_arrive_expect_tx(&bars[FULL0 + s], exp ? kStageTxExport : kStageTx);
                for (int ac = 0; ac < 2; ++ac) {
                    tma_load_2d(sp + sWQ + ac * 16384, mW, &bars[FULL0 + s], ac * 64, row);
                    if (!exp) tma_load_2d(sp + sWQ + ac * 16384 + 8192, mQt, &bars[FULL0 + s], ac * 64, row);
                    tma_load_2d(sp + sK + ac * 8192, mKt, &bars[FULL0 + s], ac * 64, row);
                }
                if (!exp) {
                    tma_load_2d(sp + sAqk, mAqk, &bars[FULL0 + s], 0, row);
                } else {  // U^T rows 0-63 and 64-127, and gamma, for the chain epilogue
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_2d(sp + sWQ + bx * 16384 + 8192, mUt, &bars[FULL0 + s], 0, (int)(ghc * kD) + 64 * bx);
                }
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
            const uint64_t dStage0 = sdesc_sw128(smem_u32(stage_ptr(0)), 16, 1024);
            const uint64_t dStageK0 = sdesc_sw128(smem_u32(stage_ptr(0) + sK), 8192, 1024);
            constexpr uint32_t kIdW = idesc_bf16(128, 64, 0, 0);   // S W^T
            constexpr uint32_t kIdO = idesc_bf16(64, 128, 0, 0);   // Q~ S^T and Aqk V_new
            constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 1);  // V_new^T K~ (K~ MN-major)
            for (int c = 0; c < nck; ++c) {
                const int s = c & 1, b = c & 1;
                const uint64_t dSt = dStage0 + (uint64_t)((s * kStage) >> 4);
                const uint64_t dK = dStageK0 + (uint64_t)((s * kStage) >> 4);
                if (!mbar_wait(&bars[FULL0 + s], (c >> 1) & 1, kPolls)) { fail(); break; }
                if (!mbar_wait(&bars[SBF], c & 1, kPolls)) { fail(); break; }
                if (*abort_flag) break;
                tc_fence_after();
                const uint32_t tDA = tDA0 + b * 64, tDO = tDO0 + b * 128;
                // the serial chain first: S W^T
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                    mma_bf16_ss(tDA, dS + off, dSt + sWQ / 16 + off, kIdW, k > 0);
                }
                mma_commit(&bars[DA1]);
                // while the state epilogue forms V_new: O = Q~ S^T (tokens as rows, M = 64), once the
                // output group has taken chunk c - 2's O out of this buffer
                if (!exp) {
                    if (c >= 2 && !mbar_wait(&bars[DOE_0 + b], ((c >> 1) - 1) & 1, kPolls)) { fail(); break; }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                        mma_bf16_ss(tDO, dSt + (sWQ + 8192) / 16 + off, dS + off, kIdO, k > 0);
                    }
                }
                if (!mbar_wait(&bars[A12], c & 1, kPolls)) { fail(); break; }
                tc_fence_after();
                // S += V_new^T K~   (TMEM S was pre-decayed by this chunk's gamma)
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_bf16_ss(tS, dA1 + k * 2, dK + k * 128, kIdS, 1);
                mma_commit(&bars[SFULL]);
                // O += Aqk V_new   (B = V_new^T rows, K-major)
                if (!exp) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) mma_bf16_ss(tDO, dSt + sAqk / 16 + k * 2, dA1 + k * 2, kIdO, 1);
                    mma_commit(&bars[DO_0 + b]);
                }
                mma_commit(&bars[EMPTY0 + s]);
            }
        }
    } else if (warp == 2) {
        // ================= export (export form only) =================
        // Per chunk c: the state's operand tile once the chain has signalled it (SBF), V_new^T once
        // it has (A12), each to the chunk's workspace slot.  Each tile is released to the chain as
        // soon as its own copy has read it; chunk c's flag is released once both of its copies are
        // written, checked after the next chunk's first copy is issued (at most one group newer).
        if (exp && lane == 0) {
            for (int c = 0; c < nck; ++c) {
                const long gh = (long)(first + c) * a.H + h;
                if (!mbar_wait(&bars[SBF], c & 1, kPolls)) { fail(); break; }
                bulk_store(a.Sx + gh * 32768, sm + oS, 32768);
                bulk_commit();
                bulk_wait_read();
                mbar_arrive(&bars[SCP]);
                if (c >= 1) {  // chunk c - 1's two copies are all but the newest group
                    asm volatile("cp.async.bulk.wait_group 1;" ::: "memory");
                    fence_proxy_async_global();
                    st_release_gpu(a.oready + gh - a.H, 1);
                }
                if (!mbar_wait(&bars[A12], c & 1, kPolls)) { fail(); break; }
                bulk_store(a.Vx + gh * 16384, sm + oA1, 16384);
                bulk_commit();
                bulk_wait_read();
                mbar_arrive(&bars[VCP]);
            }
            bulk_wait_all();
            if (nck > 0 && !*abort_flag) {
                fence_proxy_async_global();
                st_release_gpu(a.oready + (long)(first + nck - 1) * a.H + h, 1);
            }
        }
    }  // warp 3: idle
    } else if (warp < 8) {
    reg_alloc<kRegsHigh>();
    {
        // ================= state epilogue (serial chain) =================
        const int q4 = warp & 3;               // TMEM lane quarter
        const int r = q4 * 32 + lane;          // state row (d_v index) = TMEM lane
        const uint32_t lrow = static_cast<uint32_t>(q4 * 32) << 16;
        uint8_t* Sb = sm + oS;
        // initial state: S_bf16 <- S0, TMEM S <- gamma_0 S0 (32 columns at a time)
        {
            const bool row_in = r < a.d;  // rows (and columns) past the head size are zero
            const float* src = (a.initial_state && row_in) ? a.initial_state + ((long)unit * a.d + r) * a.d : nullptr;
            float* dst = (nck == 0 && a.final_state && row_in) ? a.final_state + ((long)unit * a.d + r) * a.d : nullptr;
            bool ready0 = true;
            if (nck > 0 && a.ready) ready0 = wait_ready(a.ready + (long)first * a.H + h);
            if (!ready0) fail();
            const float g0 = (nck > 0 && ready0) ? __ldg(a.scal + ((long)first * a.H + h) * 4 * kC + 3 * kC) : 0.f;
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float4 t = (src && blk * 32 < a.d) ? *reinterpret_cast<const float4*>(src + blk * 32 + j)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    f[j] = t.x; f[j + 1] = t.y; f[j + 2] = t.z; f[j + 3] = t.w;
                }
                if (nck == 0) {
                    if (dst && blk * 32 < a.d)
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(dst + blk * 32 + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                    continue;
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_sw128_chunk(Sb + (blk >> 1) * 16384, r, (blk & 1) * 4 + c8, f + 8 * c8);
                uint32_t v[32];
                if constexpr (PC) {  // first chunk's decay, one factor per key channel (column)
                    const float4* gv = reinterpret_cast<const float4*>(a.gam + ((long)first * a.H + h) * kD + blk * 32);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 t = ready0 ? __ldg(gv + j / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[j] = __float_as_uint(t.x * f[j]);
                        v[j + 1] = __float_as_uint(t.y * f[j + 1]);
                        v[j + 2] = __float_as_uint(t.z * f[j + 2]);
                        v[j + 3] = __float_as_uint(t.w * f[j + 3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(g0 * f[j]);
                }
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
        if (nck > 0 && !*abort_flag && !exp) {
            const uint4* src = reinterpret_cast<const uint4*>(a.Ut + ((long)first * a.H + h) * kD * kC + (long)r * kC);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) up_next[c8] = __ldg(src + c8);
        }
        for (int c = 0; c < nck; ++c) {
            const int b = c & 1;
            const long gh = (long)(first + c) * a.H + h;
            const bool last = (c + 1 == nck);
            // U^T row r comes straight from the workspace, loaded one chunk ahead; so does the next
            // chunk's decay
            uint4 up[8];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) up[c8] = up_next[c8];
            // the next chunk's entries (a failed wait skips them; the group leaves at its next barrier);
            // the export form takes them from the stages instead, off the chain
            const bool nready = !last && !exp && (!a.ready || wait_ready(a.ready + gh + a.H));
            if (!last && !exp && !nready) fail();
            float gnext = (!nready || PC) ? 1.0f : __ldg(a.scal + (gh + a.H) * 4 * kC + 3 * kC);
            float* gvec = reinterpret_cast<float*>(sm + oGam) + ((c + 1) & 1) * kD;
            if (PC && nready) gvec[r] = __ldg(a.gam + (gh + a.H) * kD + r);  // read after the next group barrier
            if (nready) {
                const uint4* src = reinterpret_cast<const uint4*>(a.Ut + (gh + a.H) * kD * kC + (long)r * kC);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) up_next[c8] = __ldg(src + c8);
            }
            // A failed (timed-out) wait skips the work but still reaches the group barrier, so the
            // whole group leaves the loop together.
            bool ok = mbar_wait(&bars[DA1], c & 1, kPolls);
            if (!ok) fail();
            tc_fence_after();
            // ---- V_new^T row r = U^T row r - (S W^T) row r ----
            if (exp && c >= 1 && ok) {  // the previous chunk's V_new^T has been copied out
                ok = mbar_wait(&bars[VCP], (c - 1) & 1, kPolls);
                if (!ok) fail();
            }
            if (ok && exp) {  // U^T row r from this chunk's stage (its phase completes before the MMAs ran)
                ok = mbar_wait(&bars[FULL0 + (c & 1)], (c >> 1) & 1, kPolls);
                if (!ok) fail();
                const uint8_t* ub = stage_ptr(c & 1) + sWQ + (r >> 6) * 16384 + 8192;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) up[c8] = *reinterpret_cast<const uint4*>(ub + sw128_offset(r & 63, c8 * 8));
            }
            if (ok) {
                uint32_t v[2][32];
                tmem_ld32(tDA0 + b * 64 + lrow, v[0]);
                tmem_ld32(tDA0 + b * 64 + lrow + 32, v[1]);
                tmem_wait_ld();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float u[32];
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const uint4 q = up[4 * hf + c8];
                        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
                            u[8 * c8 + 2 * e] = f.x - __uint_as_float(v[hf][8 * c8 + 2 * e]);
                            u[8 * c8 + 2 * e + 1] = f.y - __uint_as_float(v[hf][8 * c8 + 2 * e + 1]);
                        }
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) st_sw128_chunk(sm + oA1, r, 4 * hf + c8, u + 8 * c8);
                }
            }
            fence_async_smem();
            tc_fence_before();
            if (bar_sync_or(1, 128, *abort_flag != 0)) break;
            if (r == 0) mbar_arrive(&bars[A12]);
            ok = mbar_wait(&bars[SFULL], c & 1, kPolls);
            if (!ok) fail();
            tc_fence_after();
            // ---- S: mirror as bf16 operand (signalled), then pre-decay the TMEM copy by the next
            //      chunk's gamma: the products the signal starts read the mirror and write other
            //      TMEM columns, and only the next S update reads S.  After a timed-out wait (error
            //      recorded) the loads still run, on garbage but in bounds: under a condition of
            //      their own the 128 values would go to local memory. ----
            uint32_t v[4][32];
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) tmem_ld32(tS + lrow + blk * 32, v[blk]);
            tmem_wait_ld();
            if (last) {
                if (ok && a.final_state && r < a.d) {
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        if (blk * 32 >= a.d) break;
                        float* dst = a.final_state + ((long)unit * a.d + r) * a.d + blk * 32;
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<uint4*>(dst + j) = make_uint4(v[blk][j], v[blk][j + 1], v[blk][j + 2], v[blk][j + 3]);
                    }
                }
            } else {
                if (exp && ok) {  // this chunk's state tile has been copied out
                    ok = mbar_wait(&bars[SCP], c & 1, kPolls);
                    if (!ok) fail();
                }
#pragma unroll
                for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        *reinterpret_cast<uint4*>(Sb + (blk >> 1) * 16384 + sw128_offset(r, ((blk & 1) * 4 + c8) * 8)) =
                            make_uint4(pack_bf16x2(__uint_as_float(v[blk][8 * c8]), __uint_as_float(v[blk][8 * c8 + 1])),
                                       pack_bf16x2(__uint_as_float(v[blk][8 * c8 + 2]), __uint_as_float(v[blk][8 * c8 + 3])),
                                       pack_bf16x2(__uint_as_float(v[blk][8 * c8 + 4]), __uint_as_float(v[blk][8 * c8 + 5])),
                                       pack_bf16x2(__uint_as_float(v[blk][8 * c8 + 6]), __uint_as_float(v[blk][8 * c8 + 7])));
                fence_async_smem();
                tc_fence_before();
                if (bar_sync_or(1, 128, *abort_flag != 0)) break;
                if (r == 0) mbar_arrive(&bars[SBF]);
                if (exp) {  // the next chunk's gamma, from its stage slot once the stage has landed
                    const int sn = (c + 1) & 1;
                    if (!mbar_wait(&bars[FULL0 + sn], ((c + 1) >> 1) & 1, kPolls)) fail();
                    gnext = reinterpret_cast<const float*>(sm + oGam)[sn];
                }
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gj = PC ? gvec[blk * 32 + j] : gnext;
                        v[blk][j] = __float_as_uint(__uint_as_float(v[blk][j]) * gj);
                    }
                    tmem_st32(tS + lrow + blk * 32, v[blk]);
                }
                tmem_wait_st();
            }
        }
    }
    } else {
    reg_dealloc<kRegsOut>();
    if (!exp) {  // the export form leaves the output to out_chunk
        // ================= output epilogue (O and the gate) =================
        // Two groups of four warps take alternate chunks (group 0: warps 8-11, even chunks; group 1:
        // warps 12-15, odd chunks), each with its own O buffer, z buffer and named barrier, so a
        // group has two chunk periods for one chunk.  O has tokens as rows (M = 64): token 16 q + r
        // lives in TMEM lane 32 q + r of quarter q.  A 16x256b load gives this thread rows
        // rA = 16 q + lane / 4 and rA + 8 and, in every group of 8 columns, the pair 2 (lane % 4),
        // 2 (lane % 4) + 1; the four threads of a row add their squares with two shuffles.
        const int og = (warp - 8) >> 2;
        const int q4 = warp & 3;
        const int rA = q4 * 16 + (lane >> 2);
        const int cp = 2 * (lane & 3);
        const uint32_t lrow = static_cast<uint32_t>(q4 * 32) << 16;
        const uint32_t gbar = 4u + (uint32_t)og;
        const bool leader = (q4 == 0 && lane == 0);
        // z of chunk c goes to buffer c & 1 (this group's); it is requested two chunks ahead
        auto issue_z = [&](int cz) {
            const int t0z = (int)(bos + (long)cz * kC);
            uint64_t* zb = &bars[ZFULL0 + (cz & 1)];
            mbar_arrive_expect_tx(zb, 32768);
            for (int cb = 0; cb < 4; ++cb)
                tma_load_3d(sm + oZ + (cz & 1) * 32768 + cb * 8192, mZ, zb, cb * 32, h, t0z);
        };
        if (a.z && leader && og < nck) issue_z(og);
        for (int c = og; c < nck; c += 2) {
            const int b = c & 1;
            const long t0 = bos + (long)c * kC;
            const int L = (eos - t0 < kC) ? (int)(eos - t0) : kC;
            uint8_t* zt = sm + oZ + b * 32768;
            bool ok = mbar_wait(&bars[DO_0 + b], (c >> 1) & 1, kPolls);
            if (!ok) fail();
            tc_fence_after();
            uint32_t v[64];
            if (ok) {
                tmem_ld16x256b_x16(tDO0 + b * 128 + lrow, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = 0u;
            }
            float* o = reinterpret_cast<float*>(v);   // o[4 j + {0,1}]: row rA, o[4 j + {2,3}]: row rA + 8
            float ssA, ssB;
            out_sumsq(o, ssA, ssB);
            tc_fence_before();
            if (bar_sync_or(gbar, 128, *abort_flag != 0)) break;
            if (leader) mbar_arrive(&bars[DOE_0 + b]);
            if (a.z) {
                ok = mbar_wait(&bars[ZFULL0 + b], (c >> 1) & 1, kPolls);
                if (!ok) fail();
            }
            out_gate_store(o, ssA, ssB, rA, cp, zt, ok, L, t0, h, leader, gbar, mOut, a);
            // every row has read its z and written its output: the buffers may be reused once the
            // tensor store issued from the z buffer has read it
            if (bar_sync_or(gbar, 128, *abort_flag != 0)) break;
            if (leader) {
                bulk_wait_read();
                if (a.z && c + 2 < nck) issue_z(c + 2);
            }
        }
        if (leader) bulk_wait_all();  // output tensor stores complete before the CTA exits
        // a z tile still in flight (only after a timeout) must land before the CTA exits; its
        // completion is the one phase nobody waited for, so any completion state will do
        if (a.z && leader && *abort_flag) {
            for (int ph = 0; ph < 2; ++ph) mbar_wait(&bars[ZFULL0 + og], ph, 1000000u);
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

template <bool PC>
__global__ void __launch_bounds__(st::kThreads, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap mQt, const __grid_constant__ CUtensorMap mKt,
                   const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mAqk,
                   const __grid_constant__ CUtensorMap mZ, const __grid_constant__ CUtensorMap mOut, TcArgs a) {
    extern __shared__ uint8_t smraw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so that the compiler
    // keeps the shared address space (plain shared loads and stores, not generic ones)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const int unit = a.seq_order[blockIdx.x / a.H] * a.H + blockIdx.x % a.H;  // longest sequences first
    state_unit<PC, false>(sm, unit, &mQt, &mKt, &mW, &mAqk, &mZ, &mOut, &mW, a);  // no export: mUt unused
}


// ---- 3b. the outputs from the exported state (fused kernel, export form) -------------------------
//
// O = Q~ S^T + Aqk V_new for every chunk, then the gate and the stores, by a set of output CTAs (as
// many as serial passes), each chunk after its serial pass has exported the chunk's state tile and
// V_new^T (workspace flag), so that the outputs trail the serial passes while the exports are still
// in L2.  The products are the serial pass's own (same operands, same order) and the epilogue is the
// same function, so both forms give the same bits.  An output CTA's 16 warps form a pipeline over
// two item buffers (tiles) and two TMEM accumulators: warp 0 lane 0 takes items position by position
// and loads them, warp 1 lane 0 issues the products, warps 8-11 and 12-15 take alternate items
// through the gate and the stores.
namespace oc {
constexpr uint32_t oS = 0, oV = 32768, oQ = 49152, oA = 65536, oZ = 73728;  // within one item buffer
constexpr uint32_t kBuf = oZ + 32768;
constexpr uint32_t kTx = 32768 + 16384 + 16384 + 8192;
enum { FULL0 = 0, FULL1, ZF0, ZF1, OF0, OF1, OE0, OE1, EMPTY0, EMPTY1, NBAR };
struct Slot {  // the item in a buffer: chunk-head pair (-1: no more), first token, tokens, head
    long gh, t0;
    int L, h;
};
constexpr uint32_t kEngBytes = 8 * NBAR + 2 * sizeof(Slot);  // barriers, then the two buffers' items
}  // namespace oc

// All 512 threads of an output CTA; `eng` holds the engine's barriers and item slots, `tm` the
// CTA's 256 TMEM columns.  The output CTAs take the items in turn (CTA e of E takes items e,
// e + E, ...; items are position-major).  The producer waits for an item's flags before it waits
// for a free buffer, so that the two latencies overlap.  It marks the slot after the last item, and
// the one after that, with -1, which ends the MMA thread and both epilogue groups.  Waits are
// bounded; a timeout is recorded and ends the role.
__device__ __forceinline__ void out_engine(uint8_t* sm, uint8_t* eng, uint32_t tm, int n_units, int e, int E,
                                           const CUtensorMap* mQt, const CUtensorMap* mAqk, const CUtensorMap* mZ,
                                           const CUtensorMap* mOut, const TcArgs& a) {
    using namespace oc;
    uint64_t* bars = reinterpret_cast<uint64_t*>(eng);
    volatile Slot* ring = reinterpret_cast<volatile Slot*>(eng + 8 * NBAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long n_items = (long)a.n_chunks[1] * n_units;
    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {  // ---- producer ----
            long k = 0, j = e;
            bool ok = true;
            for (;; ++k) {
                const int b = (int)(k & 1);
                uint8_t* buf = sm + b * kBuf;
                // the next item whose sequence reaches its position, and where it lies
                Slot sl{-1, 0, 0, 0};
                for (; j < n_items; j += E) {
                    const int pos = (int)(j / n_units), unit = (int)(j % n_units);
                    const int nn = unit / a.H;
                    const int first = a.chunk_first[nn];
                    if (pos < a.chunk_first[nn + 1] - first) {
                        long bos, eos;
                        seq_bounds(a, nn, bos, eos);
                        sl.gh = (long)(first + pos) * a.H + unit % a.H;
                        sl.t0 = bos + (long)pos * kC;
                        sl.L = (eos - sl.t0 < kC) ? (int)(eos - sl.t0) : kC;
                        sl.h = unit % a.H;
                        j += E;
                        break;
                    }
                }
                if (sl.gh >= 0 && (!wait_ready(a.ready + sl.gh) || !wait_ready(a.oready + sl.gh))) { ok = false; break; }
                if (k >= 2 && !mbar_wait(&bars[EMPTY0 + b], ((k >> 1) - 1) & 1, kPolls)) { ok = false; break; }
                ring[b].gh = sl.gh;
                ring[b].t0 = sl.t0;
                ring[b].L = sl.L;
                ring[b].h = sl.h;
                if (sl.gh < 0) {
                    mbar_arrive(&bars[FULL0 + b]);
                    break;
                }
                fence_proxy_async_global();  // the entries and exports were written before their flags
                if (a.z) {
                    mbar_arrive_expect_tx(&bars[ZF0 + b], 32768);
                    for (int cb = 0; cb < 4; ++cb) tma_load_3d(buf + oZ + cb * 8192, mZ, &bars[ZF0 + b], cb * 32, sl.h, (int)sl.t0);
                }
                mbar_arrive_expect_tx(&bars[FULL0 + b], kTx);
                const int row = (int)(sl.gh * kC);
                for (int ac = 0; ac < 2; ++ac) tma_load_2d(buf + oQ + ac * 8192, mQt, &bars[FULL0 + b], ac * 64, row);
                tma_load_2d(buf + oA, mAqk, &bars[FULL0 + b], 0, row);
                bulk_load(buf + oS, a.Sx + sl.gh * 32768, 32768, &bars[FULL0 + b]);
                bulk_load(buf + oV, a.Vx + sl.gh * 16384, 16384, &bars[FULL0 + b]);
            }
            if (ok) {  // the slot after the last: its previous item must be done first
                const int b = (int)((k + 1) & 1);
                if (k >= 1 && !mbar_wait(&bars[EMPTY0 + b], ((k - 1) >> 1) & 1, kPolls)) ok = false;
                ring[b].gh = -1;
                mbar_arrive(&bars[FULL0 + b]);
            }
            if (!ok) record_error(a.err, GDN_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---- products: O (tokens as rows, M = 64) = Q~ S^T + Aqk V_new ----
            constexpr uint32_t kIdO = idesc_bf16(64, 128, 0, 0);
            int ends = 0;
            for (long k = 0; ends < 2; ++k) {
                const int b = (int)(k & 1);
                if (!mbar_wait(&bars[FULL0 + b], (k >> 1) & 1, kPolls)) { record_error(a.err, GDN_ERR_TIMEOUT); break; }
                if (ring[b].gh < 0) {
                    ++ends;
                    continue;
                }
                if (k >= 2 && !mbar_wait(&bars[OE0 + b], ((k >> 1) - 1) & 1, kPolls)) {
                    record_error(a.err, GDN_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                uint8_t* buf = sm + b * kBuf;
                const uint64_t dS = sdesc_sw128(smem_u32(buf + oS), 16, 1024);
                const uint64_t dV = sdesc_sw128(smem_u32(buf + oV), 16, 1024);
                const uint64_t dQ = sdesc_sw128(smem_u32(buf + oQ), 16, 1024);
                const uint64_t dA = sdesc_sw128(smem_u32(buf + oA), 16, 1024);
                const uint32_t tO = tm + (uint32_t)b * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ss(tO, dQ + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                                dS + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), kIdO, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(tO, dA + kk * 2, dV + kk * 2, kIdO, 1);
                mma_commit(&bars[OF0 + b]);
            }
        }
    } else if (warp >= 8) {  // ---- epilogue groups: group g takes the items k = g, g + 2, ... ----
        const int g = (warp - 8) >> 2, q4 = warp & 3;
        const int rA = q4 * 16 + (lane >> 2), cp = 2 * (lane & 3);
        const bool leader = q4 == 0 && lane == 0;
        const uint32_t ebar = 5u + (uint32_t)g;
        uint8_t* buf = sm + g * kBuf;
        for (long k = g;; k += 2) {
            bool ok = mbar_wait(&bars[FULL0 + g], (k >> 1) & 1, kPolls);
            const long gh = ok ? ring[g].gh : -1;
            if (!ok) record_error(a.err, GDN_ERR_TIMEOUT);
            if (gh < 0) break;
            const long t0 = ring[g].t0;
            const int L = ring[g].L, h = ring[g].h;
            ok = mbar_wait(&bars[OF0 + g], (k >> 1) & 1, kPolls);
            tc_fence_after();
            uint32_t v[64];
            tmem_ld16x256b_x16(tm + (uint32_t)g * 128 + (static_cast<uint32_t>(q4 * 32) << 16), v);  // in bounds
            tmem_wait_ld();
            tc_fence_before();
            bar_sync(ebar, 128);
            if (leader) mbar_arrive(&bars[OE0 + g]);  // O is out of TMEM: the accumulator may take item k + 2
            float* o = reinterpret_cast<float*>(v);
            float ssA, ssB;
            out_sumsq(o, ssA, ssB);
            if (a.z) ok = mbar_wait(&bars[ZF0 + g], (k >> 1) & 1, kPolls) && ok;
            if (!ok) record_error(a.err, GDN_ERR_TIMEOUT);
            out_gate_store(o, ssA, ssB, rA, cp, buf + oZ, ok, L, t0, h, leader, ebar, mOut, a);
            if (leader) bulk_wait_read();  // the staged rows have left the buffer
            bar_sync(ebar, 128);           // every row has read its z
            if (leader) mbar_arrive(&bars[EMPTY0 + g]);
        }
        if (leader) bulk_wait_all();  // output stores complete before the CTA exits
    }
}

// ---- 4. fused preparation + serial pass (few units) ----------------------------------------------
//
// With few (sequence, head) units the serial pass occupies few SMs, yet it can only start after the
// whole preparation kernel.  The fused kernel runs both in one cooperative launch (one CTA per SM,
// all resident at once): CTAs 0 .. n_units-1 each run the serial pass of one unit; every other CTA
// prepares chunks, two at a time with a decay per head (two groups of eight warps, prep2_chunk) and
// three at a time with a decay per key channel (one per warpgroup, prep_chunk), each with its own
// shared region, 128 TMEM columns and named barriers.  They take chunks from a global counter
// position by position (the first chunk of every unit, then the second, ...), so the serial passes
// find their next chunk ready.  A prepared chunk is published by a release store of its flag, which
// the serial pass acquires (bounded) before reading the chunk's entries.  Preparing CTAs never wait
// for serial ones.
namespace fz {
constexpr uint32_t kPrepStride = (prep::kBytes + 1023u) & ~1023u;
constexpr int kInst = 3;                          // chunk preparations per preparing CTA
constexpr uint32_t oTmemBase = kInst * kPrepStride;  // prep role: TMEM base address
constexpr uint32_t oItem = oTmemBase + 16;        // prep role: work item of each warpgroup
constexpr uint32_t kPrepBytes = oItem + 8 * kInst;
// decay per head: two eight-warp preparations
constexpr uint32_t kPrepStride2 = (p2::kBytes + 1023u) & ~1023u;
constexpr uint32_t oTmemBase2 = 2 * kPrepStride2;
constexpr uint32_t oItem2 = oTmemBase2 + 16;
constexpr uint32_t oEng = oItem2 + 16;            // export form: the output engine's barriers and items
constexpr uint32_t kPrepBytes2 = oEng + oc::kEngBytes;
static_assert(2 * oc::kBuf <= oTmemBase2, "the output engine's buffers within the preparations' regions");
constexpr uint32_t kPrepMax = kPrepBytes > kPrepBytes2 ? kPrepBytes : kPrepBytes2;
constexpr uint32_t kSmem = st::kSmem > kPrepMax + 1024 ? st::kSmem : kPrepMax + 1024;
static_assert(kSmem <= 232448, "fused kernel shared memory exceeds the per-block limit");
// register split of the prep role (launched at 128 per thread, 512 x 128 = 65536):
// three preparing warpgroups at 160 and the fourth at 24: 3 x 128 x 160 + 128 x 24 = 64512
constexpr int kRegsPrep = 160, kRegsIdle = 24;
static_assert(kInst * 128 * kRegsPrep + (4 - kInst) * 128 * kRegsIdle <= st::kThreads * 128,
              "register split above the launch total");
}  // namespace fz

template <bool PC, bool EXP>
__global__ void __launch_bounds__(st::kThreads, 1)
chunk_fused_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mQt,
                   const __grid_constant__ CUtensorMap mKt, const __grid_constant__ CUtensorMap mW,
                   const __grid_constant__ CUtensorMap mAqk, const __grid_constant__ CUtensorMap mZ,
                   const __grid_constant__ CUtensorMap mOut, const __grid_constant__ CUtensorMap mUt, TcArgs a,
                   int n_units) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    if ((int)blockIdx.x < n_units) {
        state_unit<PC, EXP>(sm, blockIdx.x, &mQt, &mKt, &mW, &mAqk, &mZ, &mOut, &mUt, a);
        return;
    }
    using namespace fz;
    if constexpr (!PC) {
        const int tid = threadIdx.x, warp = tid >> 5, inst = tid >> 8, ltid = tid & 255;
        uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oTmemBase2);
        volatile long* item_slot = reinterpret_cast<volatile long*>(sm + oItem2);
        if (tid == 0) {
            for (int i = 0; i < 2; ++i) {
                uint64_t* b = reinterpret_cast<uint64_t*>(sm + i * kPrepStride2 + p2::oBar);
                for (int j = 0; j < 3; ++j) mbar_init(&b[j], 1);
            }
            fence_mbar_init();
            prefetch_tmap(&mQ);
            prefetch_tmap(&mK);
            prefetch_tmap(&mV);
        }
        if (warp == 0) {
            tmem_alloc(tbase, 2 * p2::kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tm = *tbase;
        if constexpr (EXP) {
            // export form: CTAs n_units .. 2 n_units - 1 form the chunks' outputs from the start, so
            // that they trail the serial passes while the exports are still in L2; the rest prepare
            if ((int)blockIdx.x < 2 * n_units) {
                out_engine(sm, sm + oEng, tm, n_units, (int)blockIdx.x - n_units, n_units, &mQt, &mAqk, &mZ, &mOut, a);
                tc_fence_before();
                __syncthreads();
                if (warp == 0) {
                    tc_fence_after();
                    tmem_dealloc(tm, 2 * p2::kTmemCols);
                }
                return;
            }
        }
        uint8_t* smi = sm + inst * kPrepStride2;
        uint64_t* bars = reinterpret_cast<uint64_t*>(smi + p2::oBar);
        const GroupBar gb{1u + (uint32_t)inst, (uint32_t)p2::kThreads};
        prep2_init_tiles(smi, ltid);
        const long n_items = (long)a.n_chunks[1] * n_units;
        uint32_t parity = 0;
        float x0 = 0.f, x1 = 0.f;
        // Chunks are taken one at a time, without requesting the next one's tiles early: taking an
        // item ahead would hold back an early position that a serial pass is waiting for.
        for (;;) {
            if (ltid == 0) item_slot[inst] = atomicAdd(&a.n_chunks[2], 1);
            gb.sync();
            const long item = item_slot[inst];
            gb.sync();  // the slot is rewritten only after every thread has read it
            if (item >= n_items) break;
            const int pos = (int)(item / n_units), unit = (int)(item % n_units);
            const int nn = unit / a.H, hh = unit % a.H;
            const int first = a.chunk_first[nn];
            if (pos >= a.chunk_first[nn + 1] - first) continue;  // this sequence is shorter
            const long gh = (long)(first + pos) * a.H + hh;
            const ChunkPos cur = chunk_pos(a, gh);
            if (!prep2_chunk(smi, tm + (uint32_t)inst * p2::kTmemCols, bars, parity, gb, ltid, cur, false, cur, false,
                             x0, x1, &mQ, &mK, &mV, a))
                break;
            parity ^= 1u;
            __threadfence();
            gb.sync();
            if (ltid == 0) {
                fence_proxy_async_global();
                st_release_gpu(a.ready + gh, 1);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tm, 2 * p2::kTmemCols);
        }
    } else {
        const int tid = threadIdx.x, warp = tid >> 5, wg = tid >> 7, ltid = tid & 127;
        uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + oTmemBase);
        volatile long* item_slot = reinterpret_cast<volatile long*>(sm + oItem);
        if (tid == 0) {
            for (int i = 0; i < kInst; ++i) {
                uint64_t* b = reinterpret_cast<uint64_t*>(sm + i * kPrepStride + prep::oBar);
                for (int j = 0; j < 3; ++j) mbar_init(&b[j], 1);
            }
            fence_mbar_init();
            prefetch_tmap(&mQ);
            prefetch_tmap(&mK);
            prefetch_tmap(&mV);
        }
        if (warp == 0) {
            tmem_alloc(tbase, 512);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tm = *tbase;
        if (wg < kInst) {
            reg_alloc<kRegsPrep>();
            uint8_t* smi = sm + wg * kPrepStride;
            uint64_t* bars = reinterpret_cast<uint64_t*>(smi + prep::oBar);
            const GroupBar gb{1u + 2u * (uint32_t)wg};
            const long n_items = (long)a.n_chunks[1] * n_units;
            uint32_t parity = 0;
            for (;;) {
                if (ltid == 0) item_slot[wg] = atomicAdd(&a.n_chunks[2], 1);
                gb.sync();
                const long item = item_slot[wg];
                gb.sync();  // the slot is rewritten only after every thread has read it
                if (item >= n_items) break;
                const int pos = (int)(item / n_units), unit = (int)(item % n_units);
                const int nn = unit / a.H, hh = unit % a.H;
                const int first = a.chunk_first[nn];
                if (pos >= a.chunk_first[nn + 1] - first) continue;  // this sequence is shorter
                const long gh = (long)(first + pos) * a.H + hh;
                prep_chunk<PC>(smi, tm + (uint32_t)wg * prep::kTmemCols, bars, parity, gb, ltid, gh, &mQ, &mK, &mV, a);
                parity ^= 1u;
                __threadfence();
                gb.sync();
                if (ltid == 0) {
                    fence_proxy_async_global();
                    st_release_gpu(a.ready + gh, 1);
                }
            }
        } else {
            reg_dealloc<kRegsIdle>();
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tm, 512);
        }
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

bool map_tokens(CUtensorMap* m, const void* base, int total_T, int H, int d) {
    // [total_T, H, d] bf16 -> dims (d, H, total_T), box (64, 1, 64), 128-byte swizzle; with d = 64 the
    // boxes at column 64 lie past the tensor and load as zeros
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return get_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_z(CUtensorMap* m, const float* base, int total_T, int H, int d) {
    // gate input z [total_T, H, d] fp32 -> dims (d, H, total_T), box (32, 1, 64), 128-byte swizzle
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
    cuuint32_t box[3] = {32, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return get_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, es,
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

// Whether a call with this many (sequence, head) units may take the fused kernel on the current
// device (the kernel-form setting can only narrow it), and so needs room for its exported state.
bool fused_possible(long units) {
    int dev = 0, sms = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return coop && units <= sms - 1;
}

size_t prefill_tc_workspace_bytes(int num_seqs, int total_T, int H) {
    return ws_layout(num_seqs, total_T, H, fused_possible((long)num_seqs * H)).total;
}

bool prefill_tc_supported(const PrefillArgs& a) {
    return (a.d == 128 || a.d == 64) && a.qkv_dtype == GDN_BF16 && get_encoder() != nullptr && a.total_T > 0;
}

cudaError_t launch_prefill_tc(const PrefillArgs& p, cudaStream_t s) {
    const WsLayout L = ws_layout(p.num_seqs, p.total_T, p.H, fused_possible((long)p.num_seqs * p.H));
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    TcArgs a{};
    a.cu = p.cu_seqlens; a.num_seqs = p.num_seqs; a.total_T = p.total_T; a.H = p.H; a.Hk = p.Hk; a.d = p.d;
    a.q = static_cast<const __nv_bfloat16*>(p.q);
    a.k = static_cast<const __nv_bfloat16*>(p.k);
    a.v = static_cast<const __nv_bfloat16*>(p.v);
    a.conv = p.conv;
    a.g = p.g; a.beta = p.beta; a.scale = p.scale; a.use_l2 = p.use_l2;
    a.chunk_seq = reinterpret_cast<int32_t*>(ws + L.off_map);
    a.chunk_first = reinterpret_cast<int32_t*>(ws + L.off_first);
    a.n_chunks = reinterpret_cast<int32_t*>(ws + L.off_count);
    a.seq_order = reinterpret_cast<int32_t*>(ws + L.off_order);
    a.W = reinterpret_cast<__nv_bfloat16*>(ws + L.off_W);
    a.Ut = reinterpret_cast<__nv_bfloat16*>(ws + L.off_Ut);
    a.Aqk = reinterpret_cast<__nv_bfloat16*>(ws + L.off_Aqk);
    a.scal = reinterpret_cast<float*>(ws + L.off_scal);
    a.Qt = reinterpret_cast<__nv_bfloat16*>(ws + L.off_Qt);
    a.Kt = reinterpret_cast<__nv_bfloat16*>(ws + L.off_Kt);
    a.gam = reinterpret_cast<float*>(ws + L.off_gam);
    a.initial_state = p.initial_state; a.final_state = p.final_state;
    a.z = p.z; a.w = p.w; a.eps = p.eps; a.out = p.out; a.out_dtype = p.out_dtype; a.err = p.err;

    CUtensorMap mQ, mK, mV, mW, mAqk, mQt, mKt, mZ, mOut, mUt;
    if (!map_tokens(&mQ, p.q, p.total_T, p.Hk, p.d) || !map_tokens(&mK, p.k, p.total_T, p.Hk, p.d) ||
        !map_tokens(&mV, p.v, p.total_T, p.H, p.d) || !map_rows(&mW, a.W, L.nch * kC, kD, 64) ||
        !map_rows(&mAqk, a.Aqk, L.nch * kC, kC, 64) || !map_rows(&mQt, a.Qt, L.nch * kC, kD, 64) ||
        !map_rows(&mUt, a.Ut, L.nch * kD, kC, 64) ||
        !map_rows(&mKt, a.Kt, L.nch * kC, kD, 64))
        return cudaErrorInvalidValue;
    if (p.z) {
        if (!map_z(&mZ, p.z, p.total_T, p.H, p.d)) return cudaErrorInvalidValue;
    } else {
        mZ = mQ;  // never dereferenced without a gate
    }
    if (p.out_dtype == GDN_BF16) {
        if (!map_tokens(&mOut, p.out, p.total_T, p.H, p.d)) return cudaErrorInvalidValue;
    } else {
        mOut = mQ;  // never dereferenced with an fp32 output
    }

    // the fused cooperative kernel serves calls with few (sequence, head) units: at most half the SMs
    // run serial passes, the rest prepare chunks; gdn_set_kernel_forms can turn it off
    int units = p.num_seqs * p.H, sms = 0, coop = 0, dev = 0, resident = 0;
    auto fused_fn = p.g_per_channel ? chunk_fused_kernel<true, false> : chunk_fused_kernel<false, false>;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
    const int form = prefill_fused_form();
    bool fused = coop && form != GDN_FORM_OFF && units <= (form == GDN_FORM_ON ? sms - 1 : sms / 2);
    if (fused) {
        e = cudaFuncSetAttribute(fused_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fz::kSmem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, fused_fn, st::kThreads, fz::kSmem);
        if (e != cudaSuccess) return e;
        fused = resident >= 1;
    }
    a.nch = L.nch;
    a.ready = fused ? reinterpret_cast<int32_t*>(ws + L.off_ready) : nullptr;
    // The export form (decay per head, no fused convolution, at most a third of the SMs in serial
    // passes): the fused kernel's serial passes export the state and as many other CTAs form the
    // outputs while the rest prepare.  The serial chain step shortens (no output work beside it),
    // the exports are read back from L2, and the preparing CTAs keep up.  (With the convolution the
    // preparations are heavier, and a decay per key channel keeps the four-warp preparations.)
    if (fused && L.exports && !p.g_per_channel && !p.conv.w && 3 * units <= sms) {
        a.Sx = ws + L.off_Sx;
        a.Vx = ws + L.off_Vx;
        a.oready = reinterpret_cast<int32_t*>(ws + L.off_oready);
        fused_fn = chunk_fused_kernel<false, true>;
        e = cudaFuncSetAttribute(fused_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fz::kSmem);
        if (e != cudaSuccess) return e;
    }

    chunk_map_kernel<<<1, 1024, 0, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (fused) {  // one CTA per SM, all resident (cooperative launch)
        void* args[] = {&mQ, &mK, &mV, &mQt, &mKt, &mW, &mAqk, &mZ, &mOut, &mUt, &a, &units};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_fn), dim3((unsigned)sms),
                                           dim3(st::kThreads), args, fz::kSmem, s);
    }
    auto state_fn = p.g_per_channel ? chunk_state_kernel<true> : chunk_state_kernel<false>;
    if (p.g_per_channel) {  // one CTA of four warps per chunk-head pair
        e = cudaFuncSetAttribute(chunk_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep::kSmem);
        if (e != cudaSuccess) return e;
        chunk_prep_kernel<true><<<(unsigned)L.nch, prep::kThreads, prep::kSmem, s>>>(mQ, mK, mV, a);
    } else {  // two resident CTAs of eight warps per SM, each walking the chunk-head pairs
        e = cudaFuncSetAttribute(chunk_prep2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p2::kSmem);
        if (e != cudaSuccess) return e;
        const long grid = L.nch < 2L * sms ? L.nch : 2L * sms;
        chunk_prep2_kernel<<<(unsigned)grid, p2::kThreads, p2::kSmem, s>>>(mQ, mK, mV, a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(state_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st::kSmem);
    if (e != cudaSuccess) return e;
    state_fn<<<(unsigned)((long)p.num_seqs * p.H), st::kThreads, st::kSmem, s>>>(mQt, mKt, mW, mAqk, mZ, mOut, a);
    return cudaGetLastError();
}

}  // namespace gdn
