/*
 * dflash_conv2.h — C ABI of DFlash 2's two-tap dynamic depthwise convolution
 * on one GB300 GPU.
 *
 * Blog post "DFlash 2: Keep Drafting Parallel", section "A Lightweight Local
 * Convolution": in front of and behind every attention and every feed-forward
 * sublayer the drafter applies a two-tap depthwise convolution, one tap
 * weighing the current position and the other the position before it,
 *     Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1},
 * whose coefficients are a learned base kernel plus a small correction
 * computed from the current hidden state, one correction per 16 channels. The
 * first draft position reads the last verified token's representation, each
 * later position its predecessor's; nothing carries over from one block to
 * the next.
 *
 * This library computes, for every block b and row t of X [B, S, d]:
 *     corr_{t,i}[g] = sum_j Wc[2g + i, j] * X[b, t, j]        (g = 0 .. d/16 - 1)
 *     Y[b, t, c]    = (base[0, c] + corr_{t,0}[c/16]) * X[b, t, c]
 *                   + (base[1, c] + corr_{t,1}[c/16]) * X[b, t-1, c]
 * with X[b, -1, .] = 0. A block is S rows: row 0 is the last verified token's
 * representation and rows 1 .. S-1 are the draft positions. The pages do not
 * say how the correction is computed; this library takes a linear map without
 * bias (with d = 2560 and twenty such convolutions, as in a five-layer
 * drafter, that is the pages' 16.5M added parameters).
 *
 * Conventions: as in dflash_select.h (device pointers owned by the caller,
 * row-major, bf16 as 16-bit words, asynchronous on `stream`, no aborts; a
 * non-zero status means nothing was launched and dflash_last_error() has the
 * message).
 */
#ifndef DFLASH_CONV2_H
#define DFLASH_CONV2_H

#include <stdint.h>

#include "dflash_select.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dflash_conv2_ctx *dflash_conv2_handle;

/* Borrows one convolution's weights and allocates its 4-byte device error
 * word (the only allocation).
 *   base [2, d]       bf16  base kernels of tap 0 (current row) and tap 1 (row before)
 *   Wc   [d/8, d]     bf16  correction weights; row 2g + i is tap i of channel group g
 * Both must stay valid and unchanged until dflash_conv2_destroy, and be
 * 16-byte aligned. Requires d % 64 == 0 and 64 <= d <= 16384, and an sm_103
 * GPU as the current device. Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
dflash_status dflash_conv2_init(const void *base, const void *Wc, int32_t d, dflash_conv2_handle *out);

/* Y [B, S, d] bf16 = the convolution of the blocks X [B, S, d] bf16 (both
 * 16-byte aligned; Y must not overlap X). B = 0 launches nothing. Requires
 * S >= 1 and B * S < 2^31. A pipeline wait that runs out of time (1 s) is
 * latched and reported by dflash_conv2_sync_status. Errors: INVALID_ARG,
 * CUDA. */
dflash_status dflash_conv2_run(dflash_conv2_handle h, const void *X, int32_t B, int32_t S, void *Y, void *stream);

/* Waits for `stream` and reports (then clears) the device error word:
 * DFLASH_OK or DFLASH_ERR_TIMEOUT. */
dflash_status dflash_conv2_sync_status(dflash_conv2_handle h, void *stream);

/* Frees the handle (synchronises the device first). NULL is accepted. */
dflash_status dflash_conv2_destroy(dflash_conv2_handle h);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_CONV2_H */
