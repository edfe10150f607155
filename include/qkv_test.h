/* Test hooks of libqkv.so: the device-side failure paths of the decode and
 * prefill kernels.
 *
 * Not part of the stage.  Every wait of a decode or prefill kernel on a pipeline
 * or exchange barrier is bounded (0.5 s); when it runs out the kernel sets bit 1
 * (value 2) of the device status word, lets its own copies in flight land, and
 * returns, so the context stays usable and the host learns of the failure from
 * qkv_check_device_error ("73 · D3-8 — G4 FusedQKV ported to CUDA", §3.3:
 * failures are loud, never silent).  The pages have no counterpart of these entry
 * points; they exist so that a test can make such a wait run out without faulting
 * the GPU. */
#ifndef QKV_TEST_H
#define QKV_TEST_H

#include <stdint.h>

#include "qkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One decode layer of a concat-class plan, arguments as qkv_decode_step, run on
 * a bulk-copy ring kernel with every wait limited to wait_limit_us microseconds
 * (1 .. 1000) and with the last weight copy of every CTA withheld: the consumer
 * waiting for that copy gives up, sets the device status flag 2 and returns.
 * The outputs of the rows whose copy was withheld are not written; nothing is
 * written outside the caller's buffers.  Needs 16-byte aligned x and weight rows
 * of at most 16 KB (else UNSUPPORTED).  Returns after the launch; read the flag
 * with qkv_check_device_error, which also clears it.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
qkv_status qkv_test_decode_wait_timeout(const qkv_plan* plan, const float* x, const void* w, const float* bias,
                                        const int32_t* d_pos, float* q, float* k, float* v, void* kv_k, void* kv_v,
                                        uint32_t wait_limit_us, void* stream);

/* One prefill step, arguments as qkv_prefill_step, with every wait limited to
 * wait_limit_us microseconds (1 .. 1000) and with the exchange of partial sums
 * withheld: each CTA of a cluster of 2 (the two K halves of a 128-row block) skips
 * sending its partial of the peer's tile, so the peer's wait for it runs out; the
 * CTA sets the device status flag 2 and writes none of its tile (no Y rows, no
 * cache rows).  Nothing is written outside the caller's buffers.  Needs a shape that
 * runs on clusters of 2: an even number of 64-row tiles (R / 64) and H > 64 (else
 * UNSUPPORTED), with the requirements of qkv_prefill_step.  Returns after the
 * launch; read the flag with qkv_check_device_error, which also clears it.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
qkv_status qkv_test_prefill_xchg_timeout(const qkv_plan* plan, const uint16_t* X, int32_t nt, const void* w,
                                         const float* bias, const int32_t* d_positions, float* Y, void* kv_k,
                                         void* kv_v, uint32_t wait_limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QKV_TEST_H */
