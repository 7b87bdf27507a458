/*
 * A plain C99 user of libgdn.so that needs no GPU: it includes only gdn.h, links against the
 * library and checks the host-side part of the ABI (status codes and strings, workspace sizing,
 * argument validation before any launch).  Built and run by tests/test_abi_c_consumer.py.
 * Exit status 0 = every check held; otherwise the number of failed checks.
 */
#include <stdio.h>
#include <string.h>

#include "gdn.h"

static int failures = 0;

#define CHECK(cond)                                                             \
    do {                                                                        \
        if (!(cond)) {                                                          \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond);  \
            ++failures;                                                         \
        }                                                                       \
    } while (0)

/* stand-in device pointers: non-null and 16-byte aligned; every call below must be refused (or
 * have nothing to do) before it could dereference them or hand them to CUDA */
static float fake_storage[64] __attribute__((aligned(16)));
#define DP ((void*)fake_storage)
#define FP ((float*)fake_storage)

static int chunk(const void* q, int num_seqs, int total_T, int H, int H_k, int d, gdn_dtype dt,
                 void* ws, size_t ws_bytes, void* out)
{
    return gdn_chunk_fwd(q, DP, DP, FP, FP, NULL, num_seqs, total_T, H, H_k, d, d, dt,
                         GDN_DECAY_PER_HEAD, 0.0f, 1, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                         1e-6f, out, dt, ws, ws_bytes, NULL);
}

int main(void)
{
    /* the status codes and constants a C caller switches on */
    CHECK(GDN_OK == 0 && GDN_ERR_ARG == -1 && GDN_ERR_DTYPE == -2 && GDN_ERR_CU_SEQLENS == -3);
    CHECK(GDN_ERR_WORKSPACE == -4 && GDN_ERR_LAUNCH == -5 && GDN_ERR_TIMEOUT == -6);
    CHECK(GDN_ERR_UNSUPPORTED == -7 && GDN_ERR_CUDA == -8);
    CHECK(GDN_CONV_KERNEL == 4);
    CHECK(GDN_F32 == 0 && GDN_BF16 == 1);
    CHECK(GDN_DECAY_PER_HEAD == 0 && GDN_DECAY_PER_KEY_CHANNEL == 1);

    /* every status has a text; an unknown one still gets a non-null string */
    for (int s = 0; s >= -8; --s) {
        const char* t = gdn_status_string(s);
        CHECK(t != NULL && strlen(t) > 0);
    }
    CHECK(gdn_status_string(12345) != NULL);

    /* workspace sizing is host arithmetic: positive on the tensor-core path (bf16, d = 128 or 64,
     * the same for both), zero on the CUDA-core path (fp32), and growing with the number of tokens */
    size_t w1 = gdn_chunk_fwd_workspace_size(2, 8192, 16, 128, 128, GDN_BF16);
    size_t w2 = gdn_chunk_fwd_workspace_size(2, 16384, 16, 128, 128, GDN_BF16);
    CHECK(w1 > 0 && w2 > w1);
    CHECK(gdn_chunk_fwd_workspace_size(2, 8192, 16, 128, 128, GDN_F32) == 0);
    CHECK(gdn_chunk_fwd_workspace_size(2, 8192, 16, 64, 64, GDN_BF16) == w1);
    CHECK(gdn_chunk_fwd_workspace_size(2, 8192, 16, 64, 64, GDN_F32) == 0);

    /* argument errors come back before any launch */
    CHECK(chunk(NULL, 1, 64, 2, 2, 128, GDN_F32, NULL, 0, DP) == GDN_ERR_ARG);
    CHECK(chunk(DP, 1, 64, 2, 2, 128, GDN_F32, NULL, 0, NULL) == GDN_ERR_ARG);
    CHECK(chunk(DP, 1, 64, 2, 2, 128, (gdn_dtype)7, NULL, 0, DP) == GDN_ERR_DTYPE);
    CHECK(chunk(DP, 1, 64, 2, 2, 96, GDN_F32, NULL, 0, DP) == GDN_ERR_UNSUPPORTED);
    CHECK(chunk(DP, 2, 65, 2, 2, 128, GDN_F32, NULL, 0, DP) == GDN_ERR_ARG);
    CHECK(chunk(DP, 1, 64, 6, 4, 128, GDN_F32, NULL, 0, DP) == GDN_ERR_ARG);
    CHECK(chunk(DP, 2, 8192, 16, 16, 128, GDN_BF16, NULL, 0, DP) == GDN_ERR_WORKSPACE);
    CHECK(chunk(DP, 2, 8192, 16, 16, 128, GDN_BF16, DP, w1 - 1, DP) == GDN_ERR_WORKSPACE);

    CHECK(gdn_recurrent_step(DP, DP, DP, FP, FP, NULL, 4, 2, 2, 128, 128, GDN_BF16,
                             GDN_DECAY_PER_HEAD, 0.0f, 1, NULL, NULL, NULL, NULL, NULL, 1e-6f, DP,
                             GDN_BF16, NULL) == GDN_ERR_ARG);              /* no state */
    CHECK(gdn_recurrent_step(DP, DP, DP, FP, FP, FP, 0, 2, 2, 128, 128, GDN_BF16,
                             GDN_DECAY_PER_HEAD, 0.0f, 1, NULL, NULL, NULL, NULL, NULL, 1e-6f, DP,
                             GDN_BF16, NULL) == GDN_OK);                   /* nothing to do */
    CHECK(gdn_recurrent_multi_step(DP, DP, DP, FP, FP, FP, 3, NULL, 4, 2, 2, 2, 128, 128,
                                   GDN_BF16, GDN_DECAY_PER_HEAD, 0.0f, 1, NULL, NULL, NULL, NULL,
                                   NULL, 1e-6f, DP, GDN_BF16, NULL) == GDN_ERR_ARG);
    CHECK(gdn_gate_rmsnorm_silu(DP, GDN_F32, FP, NULL, 1e-6f, DP, GDN_F32, 10, 100, NULL)
          == GDN_ERR_ARG);                                                 /* d_v % 32 != 0 */
    CHECK(gdn_decay_from_logits(NULL, FP, NULL, NULL, FP, NULL, 10, 4, NULL) == GDN_ERR_ARG);
    CHECK(gdn_chunk_fwd_noalloc(NULL, DP, DP, FP, FP, NULL, 1, 64, 2, 2, 128, 128, GDN_BF16,
                                GDN_DECAY_PER_HEAD, 0.0f, 1, NULL, NULL, NULL, NULL, NULL, NULL,
                                NULL, 1e-6f, DP, GDN_BF16, NULL) == GDN_ERR_ARG);
    CHECK(gdn_get_device_error(NULL, NULL) == GDN_ERR_ARG);
    CHECK(gdn_selftest_bounded_wait(1000000ull, NULL, NULL) == GDN_ERR_ARG);
    CHECK(gdn_selftest_bounded_wait(10ull, (int*)fake_storage, NULL) == GDN_ERR_ARG);

    if (failures == 0)
        printf("c consumer ok\n");
    return failures;
}
