/* A plain C caller of the library: host-only entry points (no device work), so it
 * runs on a machine without a GPU.  Prints one line per check; exit status 0 when
 * every check holds. */
#include <stdio.h>
#include <string.h>

#include "conv2d.h"

static int failures = 0;

static void check(int ok, const char* what)
{
    printf("%s %s\n", ok ? "ok" : "FAIL", what);
    if (!ok) ++failures;
}

int main(void)
{
    conv2d_params prm;
    memset(&prm, 0, sizeof prm);
    prm.n = 4; prm.h = 56; prm.w = 56; prm.c = 64; prm.k = 64; prm.r = 3; prm.s = 3;
    prm.stride_h = prm.stride_w = 1; prm.pad_h = prm.pad_w = 1; prm.dil_h = prm.dil_w = 1; prm.groups = 1;
    int64_t p = 0, q = 0;
    check(conv2d_fwd_output_shape(&prm, &p, &q) == CONV2D_OK && p == 56 && q == 56, "output shape 56x56");
    prm.stride_h = prm.stride_w = 2;
    check(conv2d_fwd_output_shape(&prm, &p, &q) == CONV2D_OK && p == 28 && q == 28, "output shape stride 2");
    prm.groups = 3;
    check(conv2d_fwd_output_shape(&prm, &p, &q) == CONV2D_ERR_INVALID, "groups that do not divide C rejected");
    prm.groups = 1;
    check(conv2d_fwd_workspace_bytes(&prm) >= 256, "workspace has the status block");
    check(conv2d_bwd_weight_workspace_bytes(&prm) >= 256 && conv2d_bwd_data_workspace_bytes(&prm) >= 256,
          "gradient workspaces have the status block");
    check(conv2d_fwd_host_staging_bytes(&prm) > 0, "host staging size");
    check(strlen(conv2d_strerror(CONV2D_ERR_UNSUPPORTED)) > 0 && strlen(conv2d_strerror(99)) > 0, "strerror");
    check(conv2d_last_launch_count() == 0, "no launch before any call");
    conv2d_epilogue epi = {7, 0};
    char fake[64];
    void* dev = (void*)(((uintptr_t)fake + 15) & ~(uintptr_t)15);  /* aligned, never dereferenced */
    check(conv2d_fwd_epi(&prm, dev, dev, NULL, dev, NULL, 0, NULL, NULL, &epi) == CONV2D_ERR_INVALID,
          "unknown activation rejected before any device work");
    check(conv2d_fwd_output_shape(NULL, &p, &q) == CONV2D_ERR_INVALID, "null params rejected");
    return failures ? 1 : 0;
}
