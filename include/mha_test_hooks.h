/*
 * mha_test_hooks.h -- entry points of libmha.so that exist only for its own
 * tests.  They are not part of the attention API (include/mha.h) and no
 * production caller needs them; they are kept out of that header so the
 * product interface carries no process-wide test switch.
 */
#ifndef MHA_TEST_HOOKS_H
#define MHA_TEST_HOOKS_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mha_debug_withhold_p -- test hook (not for production use).  While on, every
 * later mha_fwd launch withholds one internal pipeline signal (the first
 * probability tile of its first query tile), so the kernel's bounded wait runs
 * out: after about a second each CTA aborts, waits for its own copies and
 * tensor-core operations, frees its tensor memory and records
 * MHA_ERR_TIMEOUT, which mha_sync_status returns.  Outputs of such a launch
 * are undefined.  Off by default; process-wide.
 */
void mha_debug_withhold_p(int on);

#ifdef __cplusplus
}
#endif

#endif /* MHA_TEST_HOOKS_H */
