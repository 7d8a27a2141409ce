// Launch interface of the device code (kernels.cu) used by the C ABI (api.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "icpnn_internal.h"

namespace icpnn {

// Number of leading heap slots (top tree levels) staged in shared memory by
// the search kernels: 4096 slots = levels 0..11, 32 KB.
constexpr int kSmemSlots = 4096;

// ICP pass result: 18 doubles.
//   [0] accepted pairs, [1] non-finite source points,
//   [2..4]  sum (s - c_s), [5..7] sum (q - c_q),
//   [8..16] sum (s - c_s)_a (q - c_q)_b at 8 + 3a + b, [17] sum d2.
constexpr int kMomentSlots = 18;

// Published result of a pass (`out` of launch_icp_pass and the persistent
// kernel; may be host-mapped): kResultWords 64-bit words, each
// (result_tag(seq) << 32) | payload.  Words 2v and 2v + 1 hold slot v as a
// float-float pair (the float bits of hi, then of lo; the value is
// double(hi) + double(lo)); words 36 and 37 the low 32 bits of the pass's
// start and publish global times (0 when not recorded).  The words are
// stored with no fence and in no particular order: a reader takes the
// result once every word carries the pass's tag (an 8-byte aligned word is
// written and read whole).  Word kAbortWord holds the sequence number of a
// pass that gave up waiting for its command, stored after a system-scope
// fence.
constexpr int kResultWords = 2 * kMomentSlots + 2;
constexpr int kAbortWord = kResultWords;
// The top bit set: zeroed memory never carries a valid tag.
__host__ __device__ constexpr uint32_t result_tag(unsigned long long seq) { return static_cast<uint32_t>(seq) | 0x80000000u; }

// The moment reduction combines block partials in groups of kGroupBlocks
// (one load per thread of a 256-thread block); its counter array holds
// reduction_counter_words(grid) zeroed 32-bit words: [0] finished groups,
// [1] skipped blocks, [2 + g] finished blocks of group g.
constexpr int kGroupBlocks = 256 / kMomentSlots;
constexpr int64_t reduction_counter_words(int64_t grid) { return 2 + (grid + kGroupBlocks - 1) / kGroupBlocks; }

// Command block of a pass launched before its transform is known (host-mapped,
// written by the host): rt = R (row-major) then t; word = (seq << 1) | stop,
// stored last with release semantics.
struct alignas(16) PassCommand {
  float rt[12];
  unsigned long long word;
};

// Device copy of a command (zeroed before a registration's first pass): the
// first block of a pass to arrive (elect) alone polls the host's command and
// forwards it here as word = (seq << 2) | outcome, with rt; the other blocks
// poll this word in L2 instead of host memory.
struct alignas(16) CommandMirror {
  unsigned long long elect;
  unsigned long long word;
  float rt[12];  // at byte 16: read with 16-byte vector loads
};

// Kinds of a tagged command (the low two bits of its control word).
constexpr unsigned long long kCmdPass = 0, kCmdStop = 1, kCmdResidual = 2;

// Command of the persistent registration kernel (host-mapped, written by the
// host).  Every word carries a tag naming the pass and the command's kind in
// its high half, so that a reader can tell a complete command from one caught
// half-written without an acquire fence (which would invalidate the reader's
// L1 cache, where the persistent kernel keeps the tree from pass to pass):
// words[j] = (tag << 32) | float bits of rt[j] (R row-major, then t), with
// tag = low 32 bits of ((seq << 2) | kind) and the top bit set (zeroed memory
// never carries a valid tag); ctrl = (seq << 2) | kind: kCmdPass (a
// correspondence pass), kCmdStop (leave the kernel; no words) or kCmdResidual
// (the iteration's two residual passes, which use sequence numbers seq and
// seq + 1).  The host writes the words first, then ctrl; a run command is
// taken from its words alone.
struct alignas(16) TaggedCommand {
  unsigned long long words[12];
  unsigned long long ctrl;
};

// Device copy of the tagged commands (zeroed before the kernel starts): the
// first block to wait for a pass (elect) polls the host's command and forwards
// it here; the other blocks poll this copy in L2.  ctrl = (seq << 3) | code
// (the command's kind, or 3 = gave up waiting); t_cmd = global time (ns) at
// which the command was seen.
struct alignas(16) TaggedMirror {
  unsigned long long elect;
  unsigned long long ctrl;
  unsigned long long t_cmd;
  unsigned long long pad;
  unsigned long long words[12];
};

struct IcpPassParams {
  float R[9];
  float t[3];
  float shift_s[3];   // c_s (replaced on the device when src_bbox6 is set)
  float shift_q[3];   // c_q
  float max_d2;       // accept iff d2 <= max_d2 (float threshold equivalent to the double test)
  unsigned long long seq;  // published after the result, see launch_icp_pass
  // Non-null: R and t above are ignored; every block first waits, for at
  // most wait_ns of global time, until cmd->word names this pass's seq and
  // takes R and t from cmd->rt.  A block that finds the stop bit, a later
  // seq, or no command in time does no work; the pass then publishes nothing
  // (stop, later seq) or, if any block ran out of time, stores seq in the
  // abort word (the word after the publish word).
  const PassCommand* cmd;
  CommandMirror* mirror;
  unsigned long long wait_ns;
  // If set: the source's bounding box as ordered integers (lo xyz, hi xyz),
  // computed on the device; every kernel then takes shift_s as its centre,
  // 0.5f * (lo + hi) per axis in float32 -- the same value the host decodes
  // the moments with -- so the host need not wait for the box before it
  // launches the passes.
  const int32_t* src_bbox6;
};

constexpr unsigned long long kCommandWaitNs = 50ull * 1000 * 1000;

// Bounding box of n points as order-preserving int encodings
// (lo x, lo y, lo z, hi x, hi y, hi z); non-finite points are skipped.
cudaError_t launch_bbox(const float* xyz, int64_t n, int32_t* bbox6, cudaStream_t s);
void decode_bbox(const int32_t bbox6[6], float lo[3], float hi[3]);

// 30-bit Morton code of every point over the box in bbox6; vals = 0..n-1.
cudaError_t launch_morton(const float* xyz, int64_t n, const int32_t* bbox6, uint32_t* keys,
                          uint32_t* vals, cudaStream_t s);

// Stable LSD radix sort of (key, value) pairs on key bits [lo_bit, hi_bit)
// (8 bits per pass).  Buffers: keys/vals (input), keys_alt/vals_alt (same
// size), temp of segments * radix_temp_words(n) words.  *sorted_vals receives
// whichever value buffer holds the result.  With segments > 1 the buffers
// hold that many independent arrays of n pairs, back to back, sorted in the
// same launches.
int64_t radix_temp_words(int64_t n);
cudaError_t radix_sort(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                       uint32_t* temp, int64_t n, int lo_bit, int hi_bit, cudaStream_t s,
                       uint32_t** sorted_vals, int segments = 1);

// records[i] = (xyz[perm[i]], perm[i]) as float4; perm == nullptr -> identity.
cudaError_t launch_gather(const float* xyz, int64_t n, const uint32_t* perm, float4* records,
                          cudaStream_t s);

// Exact 1-NN of every record; writes idx/dist2 at the record's original slot.
// chunk_counter: one device word (zeroed here, on the stream) from which the
// warps take chunks of queries beyond their first.
cudaError_t launch_nn(const icpnn_tree& t, const float4* queries, int64_t n, int32_t* idx,
                      float* dist2, uint32_t* chunk_counter, cudaStream_t s);

// One fused ICP pass: transform, search, reject, reduce.  `partials` holds
// grid * kMomentSlots doubles, `counter` reduction_counter_words(grid) zeroed
// words (left zeroed), `out` kAbortWord + 1 words (may be host-mapped): the
// result, published as tagged words (see kResultWords) so that the host can
// poll it instead of synchronising the stream; a pre-launched pass that gave
// up waiting for its command stores p.seq in the abort word and nothing else.
// Sequence numbers grow pass by pass, and a pass reaches its reduction only
// after its predecessor on the stream has completed, so an abort word at or
// beyond s proves that pass s has finished, published or not.
// idx/dist2 optional.
int icp_pass_grid(const icpnn_tree& t, int64_t n);
// slot_of (optional): per source record, the record slot of its accepted
// match, or -1.  leaf_of (optional): per source record, the heap id of the
// leaf where the previous pass found its best point (0: none); the search
// starts there and overwrites it.
cudaError_t launch_icp_pass(const icpnn_tree& t, const float4* src, int64_t n,
                            const IcpPassParams& p, double* partials, uint32_t* counter,
                            double* out, int32_t* idx, float* dist2, int32_t* slot_of,
                            uint32_t* leaf_of, int grid, cudaStream_t s);

// The whole registration as one persistent, cooperatively launched kernel
// (every block resident at once): it stages the top of the tree in shared
// memory once, then loops: wait for the tagged command of pass p.seq, p.seq +
// 1, ... (bounded by p.wait_ns, see IcpPassParams), run the pass exactly as
// launch_icp_pass does with the same grid (same partition of the work, same
// reduction order, so the same bits), publish the result in `out` with the
// pass's start and end global times in the two words after the abort word,
// and wait for the next command.  With slot_of (the residual rejection) the
// correspondence passes record each record's matched slot, and a residual
// command runs the iteration's two residual passes (see
// launch_residual_pass) back to back: the first hands the 3-sigma threshold
// to the second through thr_word (a device word, the pass's tag above the
// float's bits) and publishes nothing, the second publishes in out with
// seq + 1.  A stop command (or a later sequence number) ends the
// kernel; a block that gives up waiting reports the pass aborted and leaves.  The tree is read-only for the kernel's lifetime, so the L1 cache of
// each SM keeps the part of it its queries touched in the previous pass; the
// reduction takes an acquire fence only in the blocks that finish a level.
// Returns cudaErrorCooperativeLaunchTooLarge (and launches nothing) when the
// grid cannot be resident at once.
bool registration_kernel_fits(const icpnn_tree& t, int grid);
cudaError_t launch_registration(const icpnn_tree& t, const float4* src, int64_t n, const IcpPassParams& p,
                                const TaggedCommand* cmd, TaggedMirror* mirror, double* partials,
                                uint32_t* counter, double* out, unsigned long long* thr_word,
                                int32_t* slot_of, uint32_t* leaf_of, int grid, cudaStream_t s);

// Residual pass of the residual rejection (same grid, partials, counter and
// published result layout as the ICP pass): out[0] = pairs with
// e2 <= threshold, out[1] = pairs with a match, out[2..16] = moments of the
// kept pairs, out[17] = sum of e2 over all matched pairs.  The threshold is
// p.max_d2, or *thr_in (device) when thr_in is given.  With thr_out the pass
// reduces out[1] and out[17] only, stores float_threshold(9 * out[17] /
// out[1]) at thr_out for the next pass and publishes nothing; the next pass's
// out[1] and out[17] are then the same sums, bit for bit (same per-thread
// sums, same reduction order).
cudaError_t launch_residual_pass(const icpnn_tree& t, const float4* src, const int32_t* slot_of,
                                 int64_t n, const IcpPassParams& p, double* partials,
                                 uint32_t* counter, double* out, int grid, cudaStream_t s,
                                 const float* thr_in = nullptr, float* thr_out = nullptr);

// Voxel-grid downsampling of n points (device xyz) into out (device, capacity
// n x 3); *out_n = occupied voxels.  scratch: voxel_scratch_words(n) words;
// bounds: 8 device words; total: 1 device word; host_bounds: 8 host words.
// Returns 0, or -1 when a voxel index would exceed +-2^40 (or the occupied
// index box 2^63 keys); CUDA errors in *err.
int64_t voxel_scratch_words(int64_t n);
int voxel_downsample(const float* xyz, int64_t n, float v, float* out, int64_t* out_n, uint32_t* scratch,
                     long long* bounds, unsigned long long* total, long long* host_bounds, cudaStream_t s,
                     cudaError_t* err);

// Allocation-free variant of the ICP pass (reads the caller's n x 3 source in
// place, one thread per point; all scratch in a file-scope device array of
// kNoAllocMaxBlocks partial records).  noalloc_scratch() returns that array's
// device address for the current device (looked up once per device).
constexpr int kNoAllocMaxBlocks = ICPNN_NOALLOC_MAX_POINTS / 256;
constexpr int kNoAllocMaxDevices = 64;
cudaError_t noalloc_scratch(double** out);
// Scratch offsets (in doubles) of the result record and the bounding box.
constexpr int64_t noalloc_result_offset() { return static_cast<int64_t>(kNoAllocMaxBlocks) * kMomentSlots; }
constexpr int64_t noalloc_counter_offset() { return noalloc_result_offset() + kMomentSlots; }
constexpr int64_t kNoAllocCounterDoubles = (reduction_counter_words(kNoAllocMaxBlocks) + 1) / 2;
constexpr int64_t noalloc_bbox_offset() { return noalloc_counter_offset() + kNoAllocCounterDoubles; }
cudaError_t launch_icp_pass_inplace(const icpnn_tree& t, const float* xyz, int64_t n,
                                    const IcpPassParams& p, double* scratch, int32_t* idx,
                                    float* dist2, cudaStream_t s);

}  // namespace icpnn
