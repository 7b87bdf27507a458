// gate.cu -- the gated output norm (gdn_gate_rmsnorm_silu) and the gate preparation
// (gdn_decay_from_logits).  Both are elementwise / per-row and HBM-bound.
//
// Output norm: "5. 线性注意力", "门控 RMSNorm": out = w * y * rsqrt(mean(y^2) + eps) * z * sigmoid(z),
// fp32 arithmetic, one rounding at the store.  One warp per row; each lane keeps d_v/32 values
// in registers, so y is read once.
//
// Gate preparation: "6.6 Gated DeltaNet" 6.6.3: g = -exp(A_log[h]) * softplus(a + dt_bias[h]),
// beta = sigmoid(b).  softplus is log1p(exp(x)) below a cut-off of 20 and x above it (where
// log1p(exp(x)) and x agree to fp32 rounding).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

template <int NPL>  // upper bound of the values per lane, d_v / 32
__global__ void __launch_bounds__(256) gate_kernel(GateArgs a) {
    const int npl = a.d_v >> 5;
    const int lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= a.rows) return;
    const long base = row * a.d_v;
    float y[NPL];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        y[i] = 0.f;
        if (i >= npl) continue;
        const long idx = base + lane + 32 * i;
        y[i] = a.y_dtype == GDN_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.y)[idx])
                                     : static_cast<const float*>(a.y)[idx];
        ss += y[i] * y[i];
    }
    ss = warp_sum(ss);
    const float rinv = rsqrtf(ss / a.d_v + a.eps);
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        if (i >= npl) continue;
        const int c = lane + 32 * i;
        const float z = a.z[base + c];
        const float w = a.w ? a.w[c] : 1.0f;
        store_out(a.out, base + c, a.out_dtype, w * y[i] * rinv * z * sigmoidf_(z));
    }
}

template <int NPL>
cudaError_t launch_gate_n(const GateArgs& a, cudaStream_t s) {
    const long blocks = (a.rows + 7) / 8;
    gate_kernel<NPL><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

__global__ void __launch_bounds__(256) gate_prep_kernel(GatePrepArgs a) {
    const long n = a.total_T * a.H;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int h = (int)(i % a.H);
        const float x = a.a[i] + (a.dt_bias ? a.dt_bias[h] : 0.0f);
        const float sp = x > 20.0f ? x : log1pf(expf(x));
        a.g[i] = -expf(a.A_log[h]) * sp;
        if (a.b) a.beta[i] = sigmoidf_(a.b[i]);
    }
}

}  // namespace

cudaError_t launch_gate(const GateArgs& a, cudaStream_t s) {
    const int npl = a.d_v / 32;
    if (npl <= 4) return launch_gate_n<4>(a, s);
    if (npl <= 8) return launch_gate_n<8>(a, s);
    return launch_gate_n<32>(a, s);
}

cudaError_t launch_gate_prep(const GatePrepArgs& a, cudaStream_t s) {
    const long n = a.total_T * a.H;
    long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    gate_prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
