/*
 * gdn_profile.h -- diagnostic timing hook of libgdn (not part of the compute
 * ABI; no counterpart on the StateFlow pages).
 *
 * When armed, every gdn_* compute call records one caller-created CUDA event
 * on its stream before each kernel it launches and one after the last, and
 * remembers the kernel's name, so a benchmark can time each kernel on the
 * stream it runs on. Disarmed (the default) it costs nothing.
 *
 * The hook is process-global and not thread-safe: arm it, run the calls to be
 * timed from one thread, read the marks, disarm it. Events are owned by the
 * caller (cudaEvent_t handles passed as void*). When the capacity is
 * exhausted further marks are dropped and gdn_profile_count stops growing.
 */
#ifndef GDN_PROFILE_H_
#define GDN_PROFILE_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Arm with `capacity` caller-created events (NULL / 0 disarms). Resets the count. */
void gdn_profile_arm(void** events, int capacity);

/* Number of marks recorded since arming. Mark i is events[i]; the kernel that
 * ran between mark i and mark i + 1 is gdn_profile_name(i) (NULL after the
 * last kernel of a call). */
int gdn_profile_count(void);
const char* gdn_profile_name(int i);

/* Self-check of the kernels' bounded waits (failure detection without a GPU
 * fault). Launches one CTA that waits on an mbarrier nothing ever arrives at,
 * through the same bounded wait the chain kernels use, with a limit of
 * 2^limit_log2 SM clock cycles (clamped to [10, 32]); when the wait gives up
 * the kernel records GDN_ERR_TIMEOUT in the workspace's status word and
 * returns, leaving the context usable. Read the outcome with
 * gdn_workspace_status. `workspace` is any gdn workspace (256-byte aligned).
 * Returns GDN_ERR_WORKSPACE / GDN_ERR_CUDA on a bad pointer / failed launch. */
int gdn_diag_wait_timeout(void* workspace, int limit_log2, void* stream);

/* Measurement override of how gdn_chunk_fwd / gdn_chunk_fwd_save carry out a
 * fixed-length bf16 call: split the chunk into `segments` segments at 64-token
 * block boundaries (1 = no split, 0 = the library's default) and overlap the
 * Pre kernel of each segment with the state-transition chain of the previous
 * one (the StateFlow review's split-and-overlap of the state transition with
 * the dense kernels, split fraction f); with two segments the first covers
 * first_permille / 1000 of the blocks (0 = half). chain_rg = 16-value-column
 * groups per chain CTA (1 or 2; 0 = default). Results are bit-identical for
 * every setting. Process-global and not thread-safe, like the timing hook. */
void gdn_diag_set_fwd_split(int segments, int first_permille, int chain_rg);

/* The same self-check on the status word of gdn_chunk_fwd_noalloc's scratch
 * on the current device; read the outcome with gdn_noalloc_status. */
int gdn_diag_wait_timeout_noalloc(int limit_log2, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_PROFILE_H_ */
