/* A plain C99 caller of the library: builds against include/ssm.h alone and uses only
 * entry points that need no GPU (version, status strings, workspace sizes, argument
 * checks), so the C ABI can be exercised on a host without a device. */
#include <stdio.h>
#include <string.h>

#include "ssm.h"

int main(void)
{
    ssm_scan_args a;
    ssm_scan_bwd_args g;
    size_t need = 0;
    int failures = 0;

    if (ssm_version() <= 0) { puts("bad version"); ++failures; }
    if (strcmp(ssm_status_string(SSM_OK), "ok") != 0) { puts("bad status string"); ++failures; }

    memset(&a, 0, sizeof a);
    a.batch = 8; a.seqlen = 2048; a.dim = 1536; a.dstate = 16;
    a.io_dtype = SSM_BF16; a.delta_softplus = 1;
    if (ssm_scan_workspace_size(&a, &need) != SSM_OK || need < 256) {
        puts("scan workspace size"); ++failures;
    }
    a.dstate = 65;
    if (ssm_scan_workspace_size(&a, &need) != SSM_ERR_UNSUPPORTED) {
        puts("scan N > 64 not rejected"); ++failures;
    }
    if (ssm_scan_fwd(NULL, NULL) != SSM_ERR_INVALID_ARG) { puts("null args"); ++failures; }

    memset(&g, 0, sizeof g);
    g.batch = 2; g.seqlen = 64; g.dim = 32; g.dstate = 16; g.io_dtype = SSM_F32;
    g.delta_softplus = 1;
    if (ssm_scan_bwd_workspace_size(&g, &need) != SSM_OK || need != 256 + 2 * 4 * 32 * 16 * 4) {
        puts("backward workspace size"); ++failures;
    }
    printf("c abi probe: %d failure(s)\n", failures);
    return failures != 0;
}
