// abi.cu -- the extern "C" entry points of libgdn.so: argument checks, dispatch, error word.
// Declarations and the meaning of every argument are in include/gdn.h.
#include <math.h>
#include <atomic>
#include <mutex>

#include "gdn_internal.cuh"

namespace {

// Device-side status word: kernels record the first error they see (atomicCAS from 0).
__device__ int g_gdn_device_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

// Address of the error word on the current device (looked up once per device).
int* device_error_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gdn_device_error) != cudaSuccess) {
            cudaGetLastError();  // do not leave the failure for a later launch check to report
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

bool valid_dtype(int d) { return d == GDN_F32 || d == GDN_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_size_ok(int d_k, int d_v) { return d_k == d_v && (d_k == 64 || d_k == 128); }
bool heads_ok(int H, int H_k) { return H > 0 && H_k >= 1 && H_k <= H && H % H_k == 0; }
bool valid_decay(int d) { return d == GDN_DECAY_PER_HEAD || d == GDN_DECAY_PER_KEY_CHANNEL; }

// Checks the short-convolution arguments and fills c; `rows` is the number of state rows (sequences
// or pool slots).  Decode updates may be in place only without grouped heads.
int conv_args(const float* w, const float* st_in, float* st_out, int H, int H_k, int d, long rows,
              bool decode, gdn::ConvArgs& c) {
    c = gdn::ConvArgs{};
    if (!w) return (st_in || st_out) ? GDN_ERR_ARG : GDN_OK;
    const long long dim = 2LL * H_k * d + (long long)H * d;
    if (dim > 0x7fffffffLL / 4 || (long long)rows * dim * 3 > (1LL << 40)) return GDN_ERR_ARG;
    if (decode && st_in && st_in == st_out && H_k != H) return GDN_ERR_ARG;
    c.w = w; c.state_in = st_in; c.state_out = st_out; c.dim = (int)dim;
    return GDN_OK;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH; }

std::atomic<int> g_prefill_fused_form{GDN_FORM_AUTO};
std::atomic<int> g_decode_blocks_form{GDN_FORM_AUTO};

bool valid_form(int f) { return f == GDN_FORM_AUTO || f == GDN_FORM_OFF || f == GDN_FORM_ON; }

}  // namespace

namespace gdn {
int prefill_fused_form() { return g_prefill_fused_form.load(std::memory_order_relaxed); }
int decode_blocks_form() { return g_decode_blocks_form.load(std::memory_order_relaxed); }
}  // namespace gdn

extern "C" {

const char* gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_ARG: return "GDN_ERR_ARG: invalid argument (null pointer, size or alignment)";
        case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE: unknown element type";
        case GDN_ERR_CU_SEQLENS: return "GDN_ERR_CU_SEQLENS: cu_seqlens not monotone or outside [0, total_T]";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
        case GDN_ERR_LAUNCH: return "GDN_ERR_LAUNCH: kernel launch failed";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait gave up";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: head size or option not supported";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA runtime call failed";
        default: return "unknown gdn_status";
    }
}

int gdn_set_kernel_forms(int prefill_fused, int decode_blocks) {
    if (!valid_form(prefill_fused) || !valid_form(decode_blocks)) return GDN_ERR_ARG;
    g_prefill_fused_form.store(prefill_fused, std::memory_order_relaxed);
    g_decode_blocks_form.store(decode_blocks, std::memory_order_relaxed);
    return GDN_OK;
}

int gdn_get_device_error(void* stream, int* device_status) {
    if (!device_status) return GDN_ERR_ARG;
    *device_status = GDN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    int* p = device_error_ptr();
    if (!p) return GDN_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    *device_status = v;
    return GDN_OK;
}

// The tensor-core path (bf16 q/k/v; d = 128, or d = 64 run as 128-wide tiles whose extra columns
// are zeros) keeps per-chunk intermediates (W, U^T, the decayed Q K^T, Q~, K~ and decay factors,
// about 75 KB per chunk and head) in the caller's workspace; the fp32 CUDA-core path needs none.
static bool uses_tc_path(int num_seqs, int total_T, int H, int d_k, int d_v, int qkv_dtype) {
    return qkv_dtype == GDN_BF16 && d_k == d_v && (d_k == 128 || d_k == 64) && total_T > 0 &&
           num_seqs > 0 && H > 0;
}

size_t gdn_chunk_fwd_workspace_size(int num_seqs, int total_T, int H, int d_k, int d_v,
                                    gdn_dtype qkv_dtype) {
    if (!uses_tc_path(num_seqs, total_T, H, d_k, d_v, qkv_dtype)) return 0;
    return gdn::prefill_tc_workspace_bytes(num_seqs, total_T, H);
}

int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu_seqlens, int num_seqs, int total_T, int H, int H_k,
                  int d_k, int d_v, gdn_dtype qkv_dtype, gdn_decay decay, float scale,
                  int use_qk_l2norm, const float* conv_weight, const float* conv_state_in,
                  float* conv_state_out, const float* initial_state, float* final_state,
                  const float* gate_z, const float* norm_weight, float norm_eps,
                  void* out, gdn_dtype out_dtype,
                  void* workspace, size_t workspace_bytes, void* stream) {
    if (!valid_dtype(qkv_dtype) || !valid_dtype(out_dtype)) return GDN_ERR_DTYPE;
    if (num_seqs <= 0 || total_T < 0 || !heads_ok(H, H_k) || !valid_decay(decay)) return GDN_ERR_ARG;
    if (!head_size_ok(d_k, d_v)) return GDN_ERR_UNSUPPORTED;
    if ((long long)num_seqs * H > 0x7fffffffLL) return GDN_ERR_ARG;
    if (!cu_seqlens && total_T % num_seqs != 0) return GDN_ERR_ARG;
    if (total_T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;
    if (!(norm_eps >= 0.0f) || (gate_z == nullptr && norm_weight != nullptr)) return GDN_ERR_ARG;
    const void* ptrs[] = {q, k, v, g, beta, initial_state, final_state, gate_z, norm_weight, out,
                          conv_weight, conv_state_in, conv_state_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ARG;
    gdn::ConvArgs conv;
    const int crc = conv_args(conv_weight, conv_state_in, conv_state_out, H, H_k, d_k, num_seqs, false, conv);
    if (crc != GDN_OK) return crc;
    const size_t need = gdn_chunk_fwd_workspace_size(num_seqs, total_T, H, d_k, d_v, qkv_dtype);
    if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    if (total_T == 0 && !final_state && !conv_state_out) return GDN_OK;

    gdn::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
    a.cu_seqlens = cu_seqlens; a.num_seqs = num_seqs; a.total_T = total_T; a.H = H; a.Hk = H_k;
    a.d = d_k; a.qkv_dtype = qkv_dtype; a.g_per_channel = decay == GDN_DECAY_PER_KEY_CHANNEL;
    a.conv = conv;
    a.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)d_k);
    a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.initial_state = initial_state; a.final_state = final_state;
    a.z = gate_z; a.w = norm_weight; a.eps = norm_eps; a.out = out; a.out_dtype = out_dtype;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.err = device_error_ptr();
    if (!a.err) return GDN_ERR_CUDA;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (total_T > 0 || final_state) {
        if (uses_tc_path(num_seqs, total_T, H, d_k, d_v, qkv_dtype) && gdn::prefill_tc_supported(a))
            e = gdn::launch_prefill_tc(a, st);
        else
            e = gdn::launch_prefill_simt(a, st);
    }
    // the final convolution state is written after every kernel that reads the input state
    if (e == cudaSuccess && conv.state_out) e = gdn::launch_conv_state(a, st);
    return launch_status(e);
}

static int decode_entry(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float* state, int num_slots, const int32_t* idx, int N,
                        int T, int H, int H_k, int d_k, int d_v, gdn_dtype qkv_dtype,
                        gdn_decay decay, float scale, int use_qk_l2norm, const float* conv_weight,
                        const float* conv_state_in, float* conv_state_out, const float* gate_z,
                        const float* norm_weight, float norm_eps, void* out, gdn_dtype out_dtype,
                        void* stream) {
    if (!valid_dtype(qkv_dtype) || !valid_dtype(out_dtype)) return GDN_ERR_DTYPE;
    if (N < 0 || T <= 0 || !heads_ok(H, H_k) || num_slots <= 0 || !valid_decay(decay)) return GDN_ERR_ARG;
    if (!head_size_ok(d_k, d_v)) return GDN_ERR_UNSUPPORTED;
    if ((long long)N * H > 0x7fffffffLL || (long long)N * T * H * d_k > (1LL << 40)) return GDN_ERR_ARG;
    if (!idx && num_slots < N) return GDN_ERR_ARG;
    if (N == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return GDN_ERR_ARG;
    if (!(norm_eps >= 0.0f) || (gate_z == nullptr && norm_weight != nullptr)) return GDN_ERR_ARG;
    const void* ptrs[] = {q, k, v, g, beta, state, gate_z, norm_weight, out, conv_weight,
                          conv_state_in, conv_state_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ARG;
    gdn::DecodeArgs a{};
    const int crc = conv_args(conv_weight, conv_state_in, conv_state_out, H, H_k, d_k, num_slots, true, a.conv);
    if (crc != GDN_OK) return crc;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.state = state; a.num_slots = num_slots;
    a.idx = idx; a.N = N; a.T = T; a.H = H; a.Hk = H_k; a.d = d_k; a.qkv_dtype = qkv_dtype;
    a.g_per_channel = decay == GDN_DECAY_PER_KEY_CHANNEL;
    a.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)d_k);
    a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.z = gate_z; a.w = norm_weight; a.eps = norm_eps; a.out = out; a.out_dtype = out_dtype;
    a.err = device_error_ptr();
    if (!a.err) return GDN_ERR_CUDA;
    return launch_status(gdn::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

int gdn_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                       const float* beta, float* state, int N, int H, int H_k, int d_k, int d_v,
                       gdn_dtype qkv_dtype, gdn_decay decay, float scale, int use_qk_l2norm,
                       const float* conv_weight, const float* conv_state_in, float* conv_state_out,
                       const float* gate_z, const float* norm_weight, float norm_eps,
                       void* out, gdn_dtype out_dtype, void* stream) {
    return decode_entry(q, k, v, g, beta, state, N > 0 ? N : 1, nullptr, N, 1, H, H_k, d_k, d_v,
                        qkv_dtype, decay, scale, use_qk_l2norm, conv_weight, conv_state_in,
                        conv_state_out, gate_z, norm_weight, norm_eps, out, out_dtype, stream);
}

int gdn_recurrent_multi_step(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float* state_pool, int num_slots,
                             const int32_t* state_indices, int N, int T, int H, int H_k, int d_k,
                             int d_v, gdn_dtype qkv_dtype, gdn_decay decay, float scale,
                             int use_qk_l2norm, const float* conv_weight,
                             const float* conv_state_in, float* conv_state_out,
                             const float* gate_z, const float* norm_weight, float norm_eps,
                             void* out, gdn_dtype out_dtype, void* stream) {
    return decode_entry(q, k, v, g, beta, state_pool, num_slots, state_indices, N, T, H, H_k, d_k,
                        d_v, qkv_dtype, decay, scale, use_qk_l2norm, conv_weight, conv_state_in,
                        conv_state_out, gate_z, norm_weight, norm_eps, out, out_dtype, stream);
}

int gdn_gate_rmsnorm_silu(const void* y, gdn_dtype y_dtype, const float* z,
                          const float* norm_weight, float eps, void* out, gdn_dtype out_dtype,
                          long rows, int d_v, void* stream) {
    if (!valid_dtype(y_dtype) || !valid_dtype(out_dtype)) return GDN_ERR_DTYPE;
    if (rows < 0 || d_v <= 0 || d_v % 32 != 0 || d_v > 1024 || !(eps >= 0.0f)) return GDN_ERR_ARG;
    if ((rows + 7) / 8 > 0x7fffffffL) return GDN_ERR_ARG;
    if (rows == 0) return GDN_OK;
    if (!y || !z || !out) return GDN_ERR_ARG;
    gdn::GateArgs a{};
    a.y = y; a.y_dtype = y_dtype; a.z = z; a.w = norm_weight; a.eps = eps;
    a.out = out; a.out_dtype = out_dtype; a.rows = rows; a.d_v = d_v;
    return launch_status(gdn::launch_gate(a, static_cast<cudaStream_t>(stream)));
}

int gdn_decay_from_logits(const float* a_logits, const float* A_log, const float* dt_bias,
                          const float* b, float* g_out, float* beta_out, long total_T, int H,
                          void* stream) {
    if (total_T < 0 || H <= 0) return GDN_ERR_ARG;
    if (total_T == 0) return GDN_OK;
    if (!a_logits || !A_log || !g_out || (b && !beta_out)) return GDN_ERR_ARG;
    gdn::GatePrepArgs a{};
    a.a = a_logits; a.A_log = A_log; a.dt_bias = dt_bias; a.b = b;
    a.g = g_out; a.beta = beta_out; a.total_T = total_T; a.H = H;
    return launch_status(gdn::launch_gate_prep(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
