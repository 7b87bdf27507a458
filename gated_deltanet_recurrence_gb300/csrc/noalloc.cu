// noalloc.cu -- gdn_chunk_fwd_noalloc: the chunked prefill without any caller-provided or
// library-allocated workspace.
//
// Some callers cannot allocate device memory at the point where they run the prefill: code that
// runs inside a memory-pool-owning framework without access to its allocator, a process that must
// not grow its footprint after start-up, or a host program that only holds raw pointers to
// buffers somebody else owns.  For them this entry point keeps the prefill's scratch (the chunk
// numbering and the per-chunk intermediates of the tensor-core path) in a fixed array that lives
// in the library's own device memory image: every GPU that loads libgdn.so (or, under lazy module
// loading, that first runs this entry point) holds the array until the process exits, and no call
// here allocates or frees anything.
//
// Rules of use:
//   * The array holds GDN_NOALLOC_SCRATCH_BYTES.  A call whose scratch need (what
//     gdn_chunk_fwd_workspace_size reports for the same sizes) exceeds it is rejected with
//     GDN_ERR_WORKSPACE before anything is launched.
//   * All calls share the one array per device, and it keeps whatever the last call left in it.
//     The kernels write every scratch word they later read in the same call, so nothing has to
//     start at zero; but two calls whose work overlaps on the GPU (different streams, no ordering
//     between them) race on the array.  Order such calls on one stream.
//   * The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
//     that device current).  Make that first call before any stream capture that includes it.
//     With lazy module loading the array may only be placed on the device at that first lookup;
//     if the device has no room for it, the call returns GDN_ERR_CUDA and launches nothing.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once per device.  In host
// code the name g_noalloc_scratch is only a host-side stand-in, never a device address.
void* scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            // clear the runtime's last-error slot, so the failure is not reported again by the
            // launch check of a later, unrelated call
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                     const float* beta, const int32_t* cu_seqlens, int num_seqs,
                                     int total_T, int H, int H_k, int d_k, int d_v, gdn_dtype qkv_dtype,
                                     gdn_decay decay, float scale, int use_qk_l2norm,
                                     const float* conv_weight, const float* conv_state_in,
                                     float* conv_state_out, const float* initial_state,
                                     float* final_state, const float* gate_z, const float* norm_weight,
                                     float norm_eps, void* out, gdn_dtype out_dtype, void* stream) {
    if (num_seqs <= 0 || total_T < 0 || H <= 0) return GDN_ERR_ARG;
    const size_t need = gdn_chunk_fwd_workspace_size(num_seqs, total_T, H, d_k, d_v, qkv_dtype);
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void* ws = nullptr;
    if (need > 0) {
        // Argument errors first, before the CUDA runtime is touched: gdn_chunk_fwd checks every
        // argument on the host ahead of its workspace, so without one it answers
        // GDN_ERR_WORKSPACE exactly when everything else is valid, and launches nothing.
        const int rc = gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens, num_seqs, total_T, H, H_k, d_k,
                                     d_v, qkv_dtype, decay, scale, use_qk_l2norm, conv_weight,
                                     conv_state_in, conv_state_out, initial_state, final_state,
                                     gate_z, norm_weight, norm_eps, out, out_dtype, nullptr, 0,
                                     stream);
        if (rc != GDN_ERR_WORKSPACE) return rc;
        ws = scratch_ptr();
        if (!ws) return GDN_ERR_CUDA;
    }
    return gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens, num_seqs, total_T, H, H_k, d_k, d_v, qkv_dtype,
                         decay, scale, use_qk_l2norm, conv_weight, conv_state_in, conv_state_out,
                         initial_state, final_state, gate_z, norm_weight, norm_eps, out, out_dtype, ws,
                         need > 0 ? (size_t)GDN_NOALLOC_SCRATCH_BYTES : 0, stream);
}
