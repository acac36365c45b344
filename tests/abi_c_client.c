/*
 * abi_c_client.c -- a plain C99 caller of libssm's C ABI (include/ssm.h), with no
 * CUDA header and no GPU: it exercises the entry points that are pure host
 * logic (version, error strings, plans, buffer sizes) and the argument checks
 * that every compute entry point runs before it touches the device, and prints
 * what it found as `key=value` lines for test_abi_c_client_cpu.py.
 * Exit status 0 when every check held, 1 otherwise.
 */
#include <stdio.h>
#include <string.h>

#include "ssm.h"

static int failures = 0;

static void expect(int got, int want, const char* what)
{
    if (got != want) {
        printf("FAIL %s: got %d, want %d\n", what, got, want);
        ++failures;
    }
}

static ssm_dims dims_of(int64_t batch, int64_t L, int64_t dim, int64_t N, int32_t io)
{
    ssm_dims d;
    memset(&d, 0, sizeof d);
    d.batch = batch;
    d.seqlen = L;
    d.dim = dim;
    d.dstate = N;
    d.io_dtype = io;
    return d;
}

int main(void)
{
    static const int codes[] = {SSM_OK, SSM_ERR_NULL, SSM_ERR_DIMS, SSM_ERR_DTYPE,
                                SSM_ERR_ALIGN, SSM_ERR_WORKSPACE, SSM_ERR_CUDA,
                                SSM_ERR_TIMEOUT, SSM_ERR_ALIAS};
    const int ncodes = (int)(sizeof codes / sizeof codes[0]);
    ssm_dims d = dims_of(4, 2048, 1536, 16, SSM_BF16);
    ssm_plan p;
    float dummy[4] = {0.f, 0.f, 0.f, 0.f};
    int i, j;

    printf("version=%d\n", ssm_version());

    /* every code has its own text, and an unknown code has one too */
    for (i = 0; i < ncodes; ++i) {
        const char* s = ssm_strerror(codes[i]);
        if (!s || !s[0]) {
            printf("FAIL empty text for code %d\n", codes[i]);
            ++failures;
            continue;
        }
        for (j = 0; j < i; ++j)
            if (strcmp(s, ssm_strerror(codes[j])) == 0) {
                printf("FAIL codes %d and %d share a text\n", codes[i], codes[j]);
                ++failures;
            }
    }
    if (!ssm_strerror(12345) || !ssm_strerror(12345)[0]) {
        printf("FAIL no text for an unknown code\n");
        ++failures;
    }

    /* the plan and the sizes of the b4 L2048 d1536 N16 bf16 scan */
    expect(ssm_scan_plan(&d, &p), SSM_OK, "ssm_scan_plan");
    printf("chunk_len=%lld nchunks=%lld channels_per_cta=%lld ctas=%lld kernels=%d\n",
           (long long)p.chunk_len, (long long)p.nchunks, (long long)p.channels_per_cta,
           (long long)p.ctas, p.kernels);
    printf("workspace_bytes=%zu\n", ssm_scan_workspace_bytes(&d));
    printf("checkpoint_bytes=%zu\n", ssm_scan_checkpoint_bytes(&d));
    printf("bwd_workspace_bytes=%zu\n", ssm_scan_bwd_workspace_bytes(&d));
    d.flags = SSM_FLAG_BC_PER_CHANNEL;
    printf("workspace_bytes_bc_per_channel=%zu\n", ssm_scan_workspace_bytes(&d));
    d.flags = 0;

    /* argument checks that return before any device work */
    expect(ssm_selective_scan_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL,
                                  &d, NULL),
           SSM_ERR_NULL, "scan with NULL tensors");
    expect(ssm_selective_scan_fwd(dummy, dummy, dummy, dummy, dummy, NULL, NULL, NULL, 0, dummy,
                                  NULL, NULL, NULL),
           SSM_ERR_NULL, "scan with NULL dims");
    {
        ssm_dims bad = d;
        bad.dstate = 3;
        expect(ssm_scan_plan(&bad, &p), SSM_ERR_DIMS, "dstate 3");
        expect((int)ssm_scan_workspace_bytes(&bad), 0, "workspace bytes of dstate 3");
        bad = d;
        bad.io_dtype = 7;
        expect(ssm_scan_plan(&bad, &p), SSM_ERR_DTYPE, "io_dtype 7");
        bad = d;
        bad.dim = 12; /* not a multiple of 8 for bf16 */
        expect(ssm_scan_plan(&bad, &p), SSM_ERR_ALIGN, "bf16 dim 12");
        bad = d;
        bad.flags = 4; /* an unknown flag bit */
        expect(ssm_scan_plan(&bad, &p), SSM_ERR_DIMS, "unknown flag");
        bad = d;
        bad.seqlen = -1;
        expect(ssm_scan_plan(&bad, &p), SSM_ERR_DIMS, "negative seqlen");
        bad = d;
        bad.flags = SSM_FLAG_ZOH | SSM_FLAG_BC_PER_CHANNEL;   /* one variant at a time */
        expect(ssm_selective_scan_bwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL,
                                      NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                      NULL, &bad, NULL),
               SSM_ERR_DIMS, "backward with both variants");
    }
    expect(ssm_state_update(NULL, dummy, dummy, dummy, dummy, dummy, NULL, NULL, NULL, 0, dummy,
                            &d, NULL),
           SSM_ERR_NULL, "state update with NULL state");
    expect(ssm_causal_conv1d_silu(dummy, dummy, NULL, 5, dummy, &d, NULL), SSM_ERR_DIMS,
           "conv width 5");
    expect(ssm_debug_timeout_probe(NULL, 256, 16, NULL), SSM_ERR_NULL, "probe without workspace");
    expect(ssm_debug_timeout_probe_static(0, NULL), SSM_ERR_DIMS, "static probe without polls");

    /* empty problems are no-ops that succeed without any pointer */
    {
        ssm_dims e = dims_of(0, 2048, 1536, 16, SSM_BF16);
        expect(ssm_selective_scan_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL,
                                      NULL, &e, NULL),
               SSM_OK, "empty batch");
        expect((int)ssm_scan_workspace_bytes(&e), 0, "workspace bytes of an empty batch");
    }

    printf("failures=%d\n", failures);
    return failures == 0 ? 0 : 1;
}
