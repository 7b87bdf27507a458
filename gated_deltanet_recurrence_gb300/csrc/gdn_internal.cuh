// gdn_internal.cuh -- helpers shared by the kernels of libgdn.so (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr float kL2Eps = 1e-6f;  // q/k normalisation: x * rsqrt(sum x^2 + 1e-6)

// ---- element access -------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Load N consecutive elements (N in {2, 4}) starting at p, converted to fp32.  p must be
// aligned to N elements.
template <int N>
__device__ __forceinline__ void load_vec(const float* p, float* out) {
    if constexpr (N == 4) {
        float4 t = *reinterpret_cast<const float4*>(p);
        out[0] = t.x; out[1] = t.y; out[2] = t.z; out[3] = t.w;
    } else {
        float2 t = *reinterpret_cast<const float2*>(p);
        out[0] = t.x; out[1] = t.y;
    }
}
template <int N>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float* out) {
    if constexpr (N == 4) {
        uint2 t = *reinterpret_cast<const uint2*>(p);
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&t.x);
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&t.y);
        float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        out[0] = fa.x; out[1] = fa.y; out[2] = fb.x; out[3] = fb.y;
    } else {
        __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(p);
        float2 fa = __bfloat1622float2(a);
        out[0] = fa.x; out[1] = fa.y;
    }
}

__device__ __forceinline__ void store_out(void* base, long idx, gdn_dtype dt, float x) {
    if (dt == GDN_BF16) reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
    else reinterpret_cast<float*>(base)[idx] = x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// A value rounded to the element type T (the convolution output is an activation of the q/k/v
// type: rounded once, after the SiLU, before the core uses it).
template <typename T>
__device__ __forceinline__ float round_to(float x) { return x; }
template <>
__device__ __forceinline__ float round_to<__nv_bfloat16>(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Short convolution of one channel: taps w[0..3] over (h0, h1, h2, x), oldest first, then SiLU.
__device__ __forceinline__ float conv4_silu(float4 w, float h0, float h1, float h2, float x) {
    const float c = fmaf(w.w, x, fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
    return c * sigmoidf_(c);
}

// Record a device-side status in the library's error word (first writer wins).
__device__ __forceinline__ void record_error(int* err, int status) {
    if (err) atomicCAS(err, 0, status);
}

// Kernel-form overrides set through gdn_set_kernel_forms (process-wide, GDN_FORM_AUTO by default).
int prefill_fused_form();
int decode_blocks_form();

// ---- launchers (one translation unit each; called from abi.cu after argument checks) --------

// The fused short convolution ("因果卷积"): weight [dim, 4]; states [rows, dim, 3], oldest first.
struct ConvArgs {
    const float* w;         // null: no convolution
    const float* state_in;  // null: zero history
    float* state_out;       // null: not written
    int dim;                // 2 * Hk * d + H * d
};

// One or more decode tokens per sequence; the single-token call is T = 1 with slot n for
// sequence n.  q, k are [N, T, Hk, d]; v, z, out [N, T, H, d]; g [N, T, H] or [N, T, H, d].
struct DecodeArgs {
    const void* q; const void* k; const void* v; const float* g; const float* beta;
    float* state; int num_slots; const int32_t* idx; int N, T, H, Hk, d; gdn_dtype qkv_dtype;
    int g_per_channel; float scale; int use_l2; ConvArgs conv;
    const float* z; const float* w; float eps; void* out; gdn_dtype out_dtype; int* err;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

struct GateArgs {
    const void* y; gdn_dtype y_dtype; const float* z; const float* w; float eps;
    void* out; gdn_dtype out_dtype; long rows; int d_v;
};
cudaError_t launch_gate(const GateArgs& a, cudaStream_t s);

struct GatePrepArgs {
    const float* a; const float* A_log; const float* dt_bias; const float* b;
    float* g; float* beta; long total_T; int H;
};
cudaError_t launch_gate_prep(const GatePrepArgs& a, cudaStream_t s);

struct PrefillArgs {
    const void* q; const void* k; const void* v; const float* g; const float* beta;
    const int32_t* cu_seqlens; int num_seqs, total_T, H, Hk, d; gdn_dtype qkv_dtype;
    int g_per_channel; float scale; int use_l2; ConvArgs conv;
    const float* initial_state; float* final_state;
    const float* z; const float* w; float eps; void* out; gdn_dtype out_dtype;
    void* workspace; size_t workspace_bytes; int* err;
};
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t s);

// Final short-convolution state of every sequence (after the prefill kernels, same stream).
cudaError_t launch_conv_state(const PrefillArgs& a, cudaStream_t s);

// tensor-core prefill (bf16 q/k/v, d_k = d_v = 128): workspace size, availability, launch
size_t prefill_tc_workspace_bytes(int num_seqs, int total_T, int H);
bool prefill_tc_supported(const PrefillArgs& a);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

}  // namespace gdn
