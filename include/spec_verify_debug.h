/*
 * spec_verify_debug.h -- host-only introspection exported by libspec_verify.so
 * for tests.  Not part of the verification ABI; no GPU is needed.
 */
#ifndef SPEC_VERIFY_DEBUG_H
#define SPEC_VERIFY_DEBUG_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Statistics work order of the dense persistent kernel.  For ticket t of a
 * call with B rows, gamma drafts, vocabulary V and element size es (2 or 4
 * bytes), writes out3 = (row, position, unit within the position).
 * Returns 0; SV_ERR_INVALID_ARG (1) for bad arguments or t out of range;
 * SV_ERR_UNSUPPORTED (2) if the kernel's 32-bit decode of t disagrees with
 * plain 64-bit division.
 */
int sv_debug_dense_ticket(long long t, long long B, int gamma, int V, int es, long long* out3);

#ifdef __cplusplus
}
#endif
#endif
