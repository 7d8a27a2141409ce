/* icpnn_probe.h -- measurement and test helpers of libicpnn; not part of the
 * registration path and not described by the pages.
 *
 * icpnn_probe_l2_read -- read a device buffer `repeats` times in one launch
 * with loads that bypass L1 (each SM's blocks stride over the whole buffer),
 * so that for a buffer that fits in L2 the achieved rate approaches the L2
 * read bandwidth: the ceiling of a search whose tree stays L2-resident.
 *   buf      device buffer of `bytes` bytes, 16-byte aligned, bytes a
 *            multiple of 16; only read.
 *   repeats  passes over the buffer, >= 1.
 *   sink     one device uint32 that the kernel may write (keeps the loads).
 *   stream   cudaStream_t (NULL = legacy default stream); not synchronised.
 * Time it with events on `stream`; bytes read = bytes * repeats.
 * Errors: INVALID_ARG, CUDA. */
/* icpnn_probe_command_wait -- exercise the bounded wait of a pass launched
 * before its transform is known (the pre-launched passes of icpnn_icp_align):
 * launch one fused pass over src (n x 3 float32, device or host) against the
 * uploaded tree whose blocks wait at most wait_ns (1 .. 1e9) for their
 * command, then, by mode:
 *   0  write no command: every block gives up after wait_ns;
 *   1  write the stop command: the blocks return without work;
 *   2  write the identity transform: the pass runs normally;
 * synchronise `stream`, and report what the pass published in *outcome:
 * 0 nothing, 1 its sequence number in the abort word, 2 its result.
 * Expected: 1, 0, 2.
 * Errors: INVALID_ARG, NOT_UPLOADED, CUDA, NO_MEMORY. */
/* icpnn_probe_delay_commands -- host-side fault injection for tests: on the
 * calling thread, after `skip` transform commands to pre-launched passes
 * (icpnn_icp_align) have been written normally, write each of the next
 * `count` only after sleeping delay_ns (<= 1e10).  A delay beyond the passes'
 * 50 ms wait makes a pass give up, which the registration must survive by
 * falling back to ordinary launches.  count = 0 switches it off.
 * Errors: INVALID_ARG. */
/* icpnn_probe_delay_collect -- host-side fault injection for tests: on the
 * calling thread, after `skip` reads of a pre-launched pass's result
 * (icpnn_icp_align) have started normally, start each of the next `count`
 * only after sleeping delay_ns (<= 1e10).  The sleep falls between queuing
 * pass k+1 and reading pass k, as when the host thread is descheduled or a
 * profiler serialises the launches: with a delay beyond twice the 50 ms
 * command wait, pass k+1 gives up while pass k's result is still unread.
 * The registration must still read pass k's outcome, then fall back to
 * ordinary launches.  count = 0 switches it off.
 * Errors: INVALID_ARG. */
/* icpnn_probe_read_result -- the host's reader of a pass's published result,
 * applied to caller-supplied words (no GPU needed).  A pass publishes its 18
 * sums into mapped host memory as n_words = 38 64-bit words, each carrying in
 * its high 32 bits the pass's tag (the low 32 bits of its sequence number
 * with the top bit set) above a payload: words 2v and 2v + 1 the float bits
 * of the hi and lo halves of sum v (value double(hi) + double(lo)), words 36
 * and 37 the low 32 bits of the pass's start and publish global times in ns.
 * The words reach the host in no particular order, so the reader takes the
 * result only once every word carries pass `seq`'s tag.
 *   words     host array of n_words words; only read.
 *   n_words   38 (anything else is INVALID_ARG).
 *   seq       the pass's sequence number.
 *   slots     out: 18 doubles, written only when the result is complete.
 *   pass_ms   out: (publish - start) mod 2^32 ns, in ms, written only when
 *             complete.
 *   complete  out: 1 if every word names pass seq, else 0.
 * Errors: INVALID_ARG. */
#ifndef ICPNN_PROBE_H
#define ICPNN_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int icpnn_probe_l2_read(const void* buf, int64_t bytes, int32_t repeats, uint32_t* sink, void* stream);

struct icpnn_tree;
int icpnn_probe_command_wait(const struct icpnn_tree* tree, const float* src, int64_t n, uint64_t wait_ns,
                             int32_t mode, int32_t* outcome, void* stream);
int icpnn_probe_delay_commands(int32_t skip, int32_t count, uint64_t delay_ns);
int icpnn_probe_delay_collect(int32_t skip, int32_t count, uint64_t delay_ns);
int icpnn_probe_read_result(const uint64_t* words, int64_t n_words, uint64_t seq, double* slots, float* pass_ms,
                            int32_t* complete);

#ifdef __cplusplus
}
#endif

#endif /* ICPNN_PROBE_H */
