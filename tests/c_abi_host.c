/* A plain C99 program against the library's C ABI (include/qgemm.h):
 * host-side queries and refusals only, so it runs without a GPU.  Built and
 * run by tests/test_c_abi_cpu.py. */
#include <stdio.h>
#include <string.h>
#include "qgemm.h"
int main(void) {
    /* host-only queries and refusals: no device work */
    size_t ws = qgemm_workspace_bytes(QG_F32, 0, 64, 64, 4, 32);
    int st = qgemm_nbits(NULL, QG_F32, NULL, NULL, NULL, NULL, QG_F32, 1, 64, 64, 5, 32, NULL, 0, NULL);
    printf("%zu %d %s\n", ws, st, qg_status_string(st));
    return !(ws == 0 && st == QG_ERR_UNSUPPORTED && strlen(qg_status_string(st)) > 0);
}
