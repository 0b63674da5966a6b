/* abi_layout.c - a plain C99 consumer of include/tl.h.
 *
 * Compiled by the test suite with gcc -std=c99 -Wall -Wextra -Werror (no C++
 * compiler, no CUDA headers), so it shows that the header is valid C: its
 * structures, constants and prototypes.  It prints the size and field offsets of
 * every structure of the interface, one "name value" line each, which the test
 * compares with the Python binding's ctypes mirrors. */
#include <stddef.h>
#include <stdio.h>

#include "tl.h"

#define FIELD(type, field) printf(#type "." #field " %zu\n", offsetof(type, field))

typedef void (*any_fn)(void);  /* a function pointer of any type converts to another (ISO C) */

int main(void) {
    printf("tl_config %zu\n", sizeof(tl_config));
    FIELD(tl_config, param_dtype);
    FIELD(tl_config, grad_dtype);
    FIELD(tl_config, scaler_enabled);
    FIELD(tl_config, init_scale);
    FIELD(tl_config, growth);
    FIELD(tl_config, backoff);
    FIELD(tl_config, interval);
    FIELD(tl_config, min_scale);
    FIELD(tl_config, max_scale);
    printf("tl_adamw_hp %zu\n", sizeof(tl_adamw_hp));
    FIELD(tl_adamw_hp, lr);
    FIELD(tl_adamw_hp, beta1);
    FIELD(tl_adamw_hp, beta2);
    FIELD(tl_adamw_hp, eps);
    FIELD(tl_adamw_hp, weight_decay);
    printf("tl_state %zu\n", sizeof(tl_state));
    FIELD(tl_state, S);
    FIELD(tl_state, count);
    FIELD(tl_state, t);
    FIELD(tl_state, b1p);
    FIELD(tl_state, b2p);
    printf("tl_status %zu\n", sizeof(tl_status));
    FIELD(tl_status, S);
    FIELD(tl_status, count);
    FIELD(tl_status, t);
    FIELD(tl_status, skipped);
    FIELD(tl_status, found_inf);
    FIELD(tl_status, norm);
    FIELD(tl_status, coef);
    FIELD(tl_status, sumsq);
    FIELD(tl_status, b1p);
    FIELD(tl_status, b2p);
    printf("tl_norm_result %zu\n", sizeof(tl_norm_result));
    FIELD(tl_norm_result, norm);
    FIELD(tl_norm_result, coef);
    FIELD(tl_norm_result, found_inf);
    FIELD(tl_norm_result, reserved);
    FIELD(tl_norm_result, sumsq);
    printf("tl_plan_info %zu\n", sizeof(tl_plan_info));
    FIELD(tl_plan_info, nchunks);
    FIELD(tl_plan_info, nbig);
    FIELD(tl_plan_info, ngroups);
    FIELD(tl_plan_info, seg);
    FIELD(tl_plan_info, nsmall);
    FIELD(tl_plan_info, run_big);
    FIELD(tl_plan_info, run_small);
    FIELD(tl_plan_info, split_forms);
    FIELD(tl_plan_info, fused_norm);
    /* the constants are plain integer expressions */
    printf("TL_OK %d\nTL_EINVAL %d\nTL_ECUDA %d\nTL_ESTATE %d\nTL_ENOMEM %d\n", TL_OK, TL_EINVAL, TL_ECUDA,
           TL_ESTATE, TL_ENOMEM);
    printf("TL_F32 %d\nTL_BF16 %d\nTL_F16 %d\nTL_E4M3B16 %d\n", TL_F32, TL_BF16, TL_F16, TL_E4M3B16);
    /* every prototype is referenced, so a declaration C cannot parse fails the build */
    any_fn fns[] = {
        (any_fn)&tl_create, (any_fn)&tl_destroy, (any_fn)&tl_accumulate, (any_fn)&tl_unscale_check,
        (any_fn)&tl_accumulate_many, (any_fn)&tl_unscale_check_many, (any_fn)&tl_grad_norm,
        (any_fn)&tl_local_sumsq, (any_fn)&tl_grad_norm_from, (any_fn)&tl_partition, (any_fn)&tl_plan,
        (any_fn)&tl_clip_adamw_step,
        (any_fn)&tl_set_lr_schedule, (any_fn)&tl_scaler_update, (any_fn)&tl_read_status, (any_fn)&tl_get_state,
        (any_fn)&tl_set_state, (any_fn)&tl_scale_ptr, (any_fn)&tl_loss_seed, (any_fn)&tl_num_params,
        (any_fn)&tl_num_chunks, (any_fn)&tl_unscale_norm_noalloc, (any_fn)&tl_launch_count,
        (any_fn)&tl_status_string, (any_fn)&tl_last_error,
    };
    printf("functions %zu\n", sizeof(fns) / sizeof(fns[0]));
    return 0;
}
