// conv.cu -- the carried state of the short convolution after a prefill call.
//
// "5. 线性注意力", "因果卷积(Causal Conv1d)": the convolution of a token reads the three raw
// inputs before it, so a sequence continued by a later call needs its last three raw inputs per
// channel.  They are taken from the sequence itself, or, for positions before its first token,
// from the input state (zeros when there is none).  One thread per (sequence, channel); each thread
// reads its three values before writing them, so the output may alias the input state.  This runs
// after the prefill kernels on the same stream, which have finished reading the input state.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

template <typename TIn>
__global__ void conv_state_kernel(PrefillArgs a) {
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;  // n * dim + c
    const int dim = a.conv.dim;
    if (idx >= (long)a.num_seqs * dim) return;
    const int n = (int)(idx / dim), c = (int)(idx % dim);
    long bos, eos;
    if (a.cu_seqlens) {
        bos = a.cu_seqlens[n];
        eos = a.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > a.total_T) {
            record_error(a.err, GDN_ERR_CU_SEQLENS);
            return;
        }
    } else {
        const long T = a.total_T / a.num_seqs;
        bos = (long)n * T;
        eos = bos + T;
    }
    const int qk = a.Hk * a.d;
    const TIn* src;
    long stride;
    int col;
    if (c < qk) {
        src = static_cast<const TIn*>(a.q); stride = qk; col = c;
    } else if (c < 2 * qk) {
        src = static_cast<const TIn*>(a.k); stride = qk; col = c - qk;
    } else {
        src = static_cast<const TIn*>(a.v); stride = (long)a.H * a.d; col = c - 2 * qk;
    }
    float hist[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const long t = eos - 3 + j;  // absolute token index of entry j
        hist[j] = t >= bos ? to_f32(src[t * stride + col])
                           : (a.conv.state_in ? a.conv.state_in[idx * 3 + 3 + (t - bos)] : 0.f);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) a.conv.state_out[idx * 3 + j] = hist[j];
}

}  // namespace

cudaError_t launch_conv_state(const PrefillArgs& a, cudaStream_t s) {
    const long total = (long)a.num_seqs * a.conv.dim;
    const unsigned grid = (unsigned)((total + 255) / 256);
    if (a.qkv_dtype == GDN_BF16) conv_state_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
    else conv_state_kernel<float><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
