/*
 * verify_attn_testhooks.h -- the one extra entry point of the TEST build of
 * the library, libverifyattn_testhooks.so (the same sources compiled with
 * VA_TEST_HOOKS).  The product library, libverifyattn.so, does not export it.
 *
 * It exists to exercise the bounded device-side waits and their abort path on
 * a GPU without faulting or hanging it: every wait in the split-K kernel
 * gives up after a clock budget (about two seconds), sets VA_STATUS_TIMEOUT in
 * the call's status word, drains the CTA's own copies and products, frees its
 * tensor memory and returns.  The pages have no counterpart: their answer to
 * a failing kernel is to roll the service back to its previous configuration
 * (The Checkpoint Report, "Decisions Made in This Message"); this library
 * instead reports the failure in its status word and leaves the context
 * usable.
 */
#ifndef VERIFY_ATTN_TESTHOOKS_H
#define VERIFY_ATTN_TESTHOOKS_H

#include "verify_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Sets, for the current device, a gate that the producer warps of every
 * split-K CTA wait on (a bounded wait) before their first copy: they proceed
 * once the int32 at device address `flag` is non-zero.  With a flag that
 * nothing sets, each tensor-core verify call gives up after the wait's budget
 * and returns with VA_STATUS_TIMEOUT in its status word.  NULL removes the
 * gate.  Synchronous (a copy to a device symbol); not for use during stream
 * capture.  Returns VA_OK or VA_ERR_CUDA.
 */
int va_test_set_gate(const int32_t *flag);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_TESTHOOKS_H */
