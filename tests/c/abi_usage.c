/* A C99 caller of the library: every entry point of spec_verify.h, called
 * with the argument types the header declares.  Compiled (not run) by
 * tests/test_abi.py to check that the header is plain C and complete. */
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

int use_every_entry_point(void *stream)
{
    spec_verify_ctx *ctx = NULL;
    sv_status st = spec_verify_create(&ctx, 0, 256, 7, 151936, SV_BF16);
    int32_t *i32 = NULL;
    float *f32 = NULL;
    const void *cv = NULL;
    uint64_t counts[9];
    double ms_rows = 0.0, ms_sample = 0.0;
    int runs = 0;
    st = spec_verify_run(ctx, cv, cv, i32, f32, f32, 0, 256, 7, i32, i32, stream);
    st = spec_verify_run_debug(ctx, cv, cv, i32, f32, f32, 0, 256, 7, i32, i32, stream, f32, f32, f32, f32, f32);
    st = spec_verify_tree_run(ctx, cv, cv, i32, i32, f32, f32, 0, 64, 15, i32, i32, i32, f32, f32, f32, stream);
    st = spec_verify_run_fused(ctx, cv, cv, 3584, cv, cv, 896, i32, f32, f32, 0, 256, 7, i32, i32, f32, f32, f32,
                               stream);
    st = spec_verify_lm_head_logits(cv, cv, 256, 151936, 3584, f32, stream);
    st = spec_verify_kv_commit(cv, (void *)f32, i32, i32, i32, 56, 256, 7, 2048, (size_t)1024, stream);
    st = spec_verify_acceptance_counts(ctx, counts, 9, 1);
    st = spec_verify_get_status(ctx);
    st = spec_verify_set_cluster_size(ctx, 0);
    st = (sv_status)spec_verify_cluster_size(ctx, 256, 7);
    st = spec_verify_set_fused_logits(ctx, 1);
    st = spec_verify_profile(ctx, 1);
    st = spec_verify_profile_read(ctx, &ms_rows, &ms_sample, &runs);
    st = spec_verify_run_noalloc(cv, cv, i32, f32, f32, 0, 256, 7, 151936, SV_BF16, i32, i32, stream);
    int gave_up = 0;
    st = spec_verify_selftest_timeout(1000, &gave_up, stream);
    (void)spec_verify_error_string(st);
    spec_verify_destroy(ctx);
    return (int)st + SV_KV_OVERFLOW + SV_KV_BAD_COUNT;
}
