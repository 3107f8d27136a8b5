/* Host-side checks of the C ABI from plain C: argument, shape and
 * alignment errors, sizing helpers and status strings.  Every call here
 * returns before any CUDA call, so it runs on a machine without a GPU.
 * Exit status 0 when every check passes; otherwise the first failing line
 * is printed and the status is 1. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "opw.h"

static int failures = 0;

#define EXPECT(cond)                                                 \
    do {                                                             \
        if (!(cond)) {                                               \
            printf("FAILED line %d: %s\n", __LINE__, #cond);         \
            ++failures;                                              \
        }                                                            \
    } while (0)

int main(void)
{
    /* Fake device addresses: aligned integers that validation never dereferences. */
    void* const heap = (void*)(uintptr_t)0x100000;
    void* const B = (void*)(uintptr_t)0x200000;
    void* G = (void*)(uintptr_t)0x300000;
    void* C = (void*)(uintptr_t)0x400000;
    int32_t* status = (int32_t*)(uintptr_t)0x500000;
    int64_t rank_off[2] = {0, 65536};
    opw_symm symm;
    memset(&symm, 0, sizeof symm);
    symm.heap_dev = heap;
    symm.rank_off = rank_off;
    symm.R = 2;

    EXPECT(opw_abi_version() == 2);
    EXPECT(strcmp(opw_status_str(OPW_OK), "OK") == 0);
    EXPECT(strcmp(opw_status_str(OPW_ERR_FLAG_PROTOCOL), "FLAG_PROTOCOL") == 0);

    /* sizing helpers */
    EXPECT(opw_ag_flag_tile(1024, 4096) == 128);
    EXPECT(opw_ag_flag_tile(64, 128) == 64);
    EXPECT(opw_ag_num_flags(8, 1024, 4096) == 2048);
    EXPECT(opw_ag_num_flags(9, 128, 128) == -1);
    EXPECT(opw_rs_num_flags(8, 8192, 4096) == 2048);
    EXPECT(opw_ring_num_flags(3, 3 * 400) == 3 * 4 * 1);
    EXPECT(opw_alltoall_num_flags(8, 65536) == 8 * 8 * 2);

    /* options default */
    opw_opts o;
    opw_opts_default(&o);
    EXPECT(o.sync_mode == OPW_SYNC_OVERLAP && o.role == OPW_ROLE_FUSED && o.local_rank == 0 &&
           o.tile_n == 0);
    /* pair tile width: an explicit choice is returned as is; others are refused */
    opw_opts wide = o;
    wide.tile_n = 512;
    EXPECT(opw_ag_tile_n(2, 128, 1024, &wide) == 512);
    wide.tile_n = 384;
    EXPECT(opw_ag_tile_n(2, 128, 1024, &wide) == -1);
    EXPECT(opw_ag_tile_n(0, 128, 1024, NULL) == -1);

    /* AG-GEMM argument checks, through the entry that needs no signal object */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, C, NULL, NULL, NULL) ==
           OPW_ERR_INVALID_ARG);                                   /* no status word */
    EXPECT(opw_ag_gemm_noalloc(NULL, 0, 128, 256, 256, B, G, C, status, NULL, NULL) ==
           OPW_ERR_INVALID_ARG);                                   /* no symmetric table */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 100, 256, 256, B, G, C, status, NULL, NULL) ==
           OPW_ERR_UNSUPPORTED_SHAPE);                             /* M_r not a flag-tile multiple */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 100, 256, B, G, C, status, NULL, NULL) ==
           OPW_ERR_UNSUPPORTED_SHAPE);                             /* N not a multiple of 8 */
    EXPECT(opw_ag_gemm_noalloc(&symm, 8, 128, 256, 256, B, G, C, status, NULL, NULL) ==
           OPW_ERR_MISALIGNED);                                    /* shard offset */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, (char*)C + 4, status, NULL, NULL) ==
           OPW_ERR_MISALIGNED);                                    /* C */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, C, status + 1, NULL, NULL) ==
           OPW_ERR_MISALIGNED);                                    /* status word */
    opw_opts bad = o;
    bad.local_rank = 2; /* R = 2 */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, C, status, &bad, NULL) ==
           OPW_ERR_INVALID_ARG);
    bad = o;
    bad.tile_n = 128; /* pair tiles are 256 or 512 wide */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, C, status, &bad, NULL) ==
           OPW_ERR_INVALID_ARG);
    bad = o;
    bad.role = OPW_ROLE_PRODUCER; /* the no-alloc entry runs the fused path only */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, C, status, &bad, NULL) ==
           OPW_ERR_INVALID_ARG);
    int32_t perm[2] = {1, 1};
    bad = o;
    bad.publish_perm = perm; /* not a permutation */
    EXPECT(opw_ag_gemm_noalloc(&symm, 0, 128, 256, 256, B, G, C, status, &bad, NULL) ==
           OPW_ERR_INVALID_ARG);
    int64_t odd_off[2] = {0, 65544};
    opw_symm odd = symm;
    odd.rank_off = odd_off;
    EXPECT(opw_ag_gemm_noalloc(&odd, 0, 128, 256, 256, B, G, C, status, NULL, NULL) ==
           OPW_ERR_MISALIGNED);                                    /* rank offset */
    odd = symm;
    odd.R = 0;
    EXPECT(opw_ag_gemm_noalloc(&odd, 0, 128, 256, 256, B, G, C, status, NULL, NULL) ==
           OPW_ERR_INVALID_ARG);

    /* calls that need a signal object refuse a null one */
    EXPECT(opw_ag_gemm(&symm, 0, 128, 256, 256, B, G, C, NULL, 1, NULL, NULL) == OPW_ERR_INVALID_ARG);
    EXPECT(opw_gemm_rs(&symm, 0, 0, 0, 256, 256, 128, NULL, 1, NULL, NULL) == OPW_ERR_INVALID_ARG);
    EXPECT(opw_gemm_rs_consume(&symm, 0, 0, 0, 256, 256, 128, C, NULL, 1, NULL, NULL) ==
           OPW_ERR_INVALID_ARG);
    EXPECT(opw_gemm_rs_consume(&symm, 0, 0, 0, 256, 256, 128, NULL, NULL, 1, NULL, NULL) ==
           OPW_ERR_INVALID_ARG);
    EXPECT(opw_signal_alloc(NULL, 16, NULL) == OPW_ERR_INVALID_ARG);
    EXPECT(opw_signal_free(NULL) == OPW_OK);

    if (failures == 0) printf("c_abi_checks: all passed\n");
    return failures == 0 ? 0 : 1;
}
