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
 * Work order of the dense persistent kernel.  For ticket t of a call with B
 * rows, gamma drafts, vocabulary V, element size es (2 or 4 bytes) and a lag
 * of `lag` rows between a row's statistics units and its residual units,
 * writes out3[0] = 1 for a residual unit (0 for statistics), out3[1] = the
 * row, out3[2] = the unit's index among that row's units of that kind.
 * Returns 0, or SV_ERR_INVALID_ARG (1) for bad arguments.
 */
int sv_debug_dense_ticket(long long t, long long B, int gamma, int V, int es, int lag,
                          long long* out3);

#ifdef __cplusplus
}
#endif
#endif
