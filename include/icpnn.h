/*
 * icpnn -- KD-tree nearest-neighbour search and ICP rigid registration on
 * one NVIDIA GB300 (sm_103a).  Plain C ABI: host or device pointers and
 * sizes only; no framework types cross this boundary.
 *
 * The method is the one of "Implementing ICP with CUDA-KDTree"
 * (pwwt.cn/news/5235220):
 *   - section 2.1: the objective E(R,t) = sum_i ||R s_i + t - t_i||^2, with t_i
 *     the target point nearest to R s_i + t, minimised by alternating a
 *     correspondence search and an SVD solve (centroids, cross-covariance H,
 *     SVD, rotation, translation from the centroid difference);
 *   - sections 2.2, 3.1, 4.1, 4.2, 5.1, 5.2: the target KD-tree, built once on
 *     the host (split axis of largest variance, median split, small leaves,
 *     depth cap 20) and stored as an index-linked array in device memory;
 *   - section 3.2: one exact nearest-neighbour query per source point;
 *   - sections 3.3 and 5.5: the source stays resident, every iteration
 *     transforms the original coordinates with the accumulated (R, t), only a
 *     small result crosses to the host per iteration;
 *   - section 4.4: correspondences farther than a maximum distance are
 *     dropped; section 4.6: stop once the change of the mean squared
 *     correspondence distance stays below eps for two iterations;
 *   - section 5.3: queries are reordered along a Morton curve for warp
 *     coherence.
 *
 * Conventions shared by every call
 *   - Points are row-major n x 3 float32 (x, y, z of point i at 3i, 3i+1,
 *     3i+2): the page's interleaved src[i*3] layout.
 *   - Return value: ICPNN_OK (0) or a negative icpnn_status.  No call aborts,
 *     traps, prints or throws; icpnn_last_error() returns a message for the
 *     calling thread's most recent failure.
 *   - Device pointers must be on the current CUDA device, the one the tree
 *     was uploaded to.  `stream` is a cudaStream_t passed as void* (NULL = the
 *     legacy default stream).
 *   - Nearest neighbour is exact and unique: for a query q the result is the
 *     target point j minimising (d2(q, r_j), j) lexicographically, with
 *     d2 = (dx*dx + dy*dy) + dz*dz, dx = r.x - q.x etc., every operation a
 *     correctly rounded float32 operation (no fused multiply-add).  Ties in
 *     d2 therefore go to the lowest target index, and the result does not
 *     depend on the tree's shape or the traversal order.  A query with a
 *     non-finite coordinate matches nothing: idx = -1, dist2 = NaN.
 */
#ifndef ICPNN_H
#define ICPNN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum icpnn_status {
    ICPNN_OK = 0,
    ICPNN_ERR_INVALID_ARG = -1,  /* null pointer, size or parameter out of range */
    ICPNN_ERR_NOT_UPLOADED = -2, /* tree has no device copy on the current device */
    ICPNN_ERR_CUDA = -3,         /* a CUDA runtime call failed (message has the name) */
    ICPNN_ERR_DEGENERATE = -4,   /* < 3 accepted pairs, or H of rank < 2 */
    ICPNN_ERR_TREE_DEPTH = -5,   /* requested depth cap outside 0..ICPNN_MAX_DEPTH */
    ICPNN_ERR_NONFINITE = -6,    /* NaN or Inf in a target or source coordinate */
    ICPNN_ERR_NO_MEMORY = -7     /* host or device allocation failed */
} icpnn_status;

/* Depth cap of the page's section 5.2: a node at this depth is a leaf holding
 * all its remaining points. */
#define ICPNN_MAX_DEPTH 20
#define ICPNN_MAX_LEAF_SIZE 64

/* kdtree_build flags */
#define ICPNN_SPLIT_ROUND_ROBIN 8u /* split axis x, y, z, x, ... by depth (page section 4.2) */

/* nn_query flags */
#define ICPNN_MORTON_SORT 1u /* reorder queries along a 30-bit Morton curve first */

/* icp_align flags */
#define ICPNN_TRACE_TIMING 2u     /* fill icpnn_iter_record.kernel_ms (CUDA events) */
#define ICPNN_RESIDUAL_REJECT 4u  /* page section 4.4: after each solve drop pairs whose
                                     residual exceeds 3 sigma and solve again */
#define ICPNN_NO_PRELAUNCH 16u    /* launch each pass only once its transform is solved
                                     (see icpnn_icp_align) */
#define ICPNN_NO_PERSISTENT 32u   /* pre-launch the passes one at a time instead of running
                                     the registration as one persistent kernel */

typedef struct icpnn_tree icpnn_tree; /* opaque; owned by the library */

/* ---------------------------------------------------------------- tree --
 * icpnn_kdtree_build -- build the target KD-tree on the host (page sections
 * 2.2, 2.3, 4.2, 5.1, 5.2).
 *   xyz_host   n x 3 float32 target points in host memory; copied, the caller
 *              keeps ownership.
 *   n          1 .. 2^31 - 1 points.
 *   leaf_size  1 .. ICPNN_MAX_LEAF_SIZE: a node holding at most this many
 *              points is a leaf (the page recommends 8 to 16).
 *   max_depth  0 .. ICPNN_MAX_DEPTH, or -1 for the page's 20; a node at this
 *              depth is a leaf whatever its size.
 *   flags      0, or ICPNN_SPLIT_ROUND_ROBIN for the page's alternative axis
 *              rule (section 4.2): x, y, z, x, ... by depth.
 *   out        receives the new tree; free it with icpnn_kdtree_free.
 * Split rule: axis of largest population variance (computed in double; axes
 * within a relative 1e-9 of the largest count as tied, the lowest wins),
 * median split: left holds the floor(count/2) smallest points ordered by
 * (coordinate, point index), right the rest, split value = the coordinate of
 * the smallest right point.  Nearest-neighbour results never depend on the
 * rule; only the search cost does.
 * Errors: INVALID_ARG, TREE_DEPTH, NONFINITE (any coordinate NaN/Inf),
 * NO_MEMORY.  Host only; needs no GPU. */
int icpnn_kdtree_build(const float* xyz_host, int64_t n, int32_t leaf_size, int32_t max_depth,
                       uint32_t flags, icpnn_tree** out);

/* icpnn_kdtree_build_device -- the same tree as icpnn_kdtree_build, node for
 * node (split axes, split values, leaf ranges and the set of points in each
 * leaf; only the order of points inside a leaf may differ), built on the
 * current CUDA device and left there, already uploaded.  The pages build the
 * tree on the host (section 5.1); this is for pipelines in which the host
 * build would be the longest step.
 *   xyz        n x 3 float32 target points, device or host memory (a host
 *              array is copied to the device first); the caller keeps
 *              ownership.
 *   n, leaf_size, max_depth, flags, out: as for icpnn_kdtree_build.
 *   stream     cudaStream_t (NULL = legacy default stream); synchronised
 *              before return.
 * The host copies of the nodes and records are made on first need
 * (icpnn_kdtree_export, icpnn_kdtree_upload to another device).
 * Errors: as icpnn_kdtree_build, plus CUDA. */
int icpnn_kdtree_build_device(const float* xyz, int64_t n, int32_t leaf_size, int32_t max_depth,
                              uint32_t flags, icpnn_tree** out, void* stream);

/* icpnn_kdtree_upload -- copy the tree (node array and leaf-ordered point
 * records) to the current device, enqueued on `stream`; the call returns
 * without waiting for the copies (the host arrays are page-locked when a
 * device is present).  Every later call that uses the tree orders its own
 * stream after them, so the tree may be used on any stream at once.  Done
 * once per target (page sections 2.3, 5.5).  A second call on the same device
 * is a no-op; a call on another device moves the copy.  Errors: INVALID_ARG,
 * CUDA, NO_MEMORY (a failed copy surfaces at the next call that waits). */
int icpnn_kdtree_upload(icpnn_tree* tree, void* stream);

/* icpnn_kdtree_free -- release the host and device copies (it synchronises
 * the tree's device first, so an upload still copying is finished).  NULL is
 * a no-op.  The caller must make sure no enqueued work still reads the tree. */
void icpnn_kdtree_free(icpnn_tree* tree);

/* icpnn_kdtree_info -- shape of a built tree.  Any output may be NULL.
 *   n_points, leaf_size, max_depth as built; depth = deepest node (root 0);
 *   n_nodes = number of tree nodes (inner + leaf). */
int icpnn_kdtree_info(const icpnn_tree* tree, int64_t* n_points, int32_t* leaf_size,
                      int32_t* max_depth, int32_t* depth, int64_t* n_nodes);

/* icpnn_kdtree_export -- the tree in the page's section 3.1 form, for
 * inspection: nodes in recursion (pre-)order, root at 0, each with split_val,
 * split_dim (0 x, 1 y, 2 z; -1 for leaves), left/right child (-1 for leaves)
 * and the half-open [start, end) range of its points in leaf_index;
 * leaf_index[k] = target point index of leaf slot k.  Arrays are caller-owned
 * host memory with node_capacity entries (>= n_nodes) and n_points entries
 * for leaf_index.  Errors: INVALID_ARG. */
int icpnn_kdtree_export(const icpnn_tree* tree, int64_t node_capacity, float* split_val,
                        int32_t* split_dim, int32_t* left, int32_t* right, int32_t* start,
                        int32_t* end, int32_t* leaf_index);

/* ---------------------------------------------------------------- query --
 * icpnn_nn_query -- exact 1-NN of every query among the tree's points (page
 * section 3.2, one query per source point).
 *   xyz        n x 3 float32 queries, device memory (or pinned/pageable host
 *              memory: then copied in on `stream`).
 *   idx, dist2 n outputs each (target index, squared distance), in the
 *              queries' order; device memory, or host memory (copied back on
 *              `stream`, which is then synchronised).
 *   flags      ICPNN_MORTON_SORT or 0.  Results do not depend on it.
 * Device inputs and outputs: asynchronous on `stream`; scratch memory is
 * drawn from the stream-ordered allocator and returned on the same stream.
 * n = 0 is allowed and does nothing.
 * Errors: INVALID_ARG, NOT_UPLOADED, CUDA, NO_MEMORY. */
int icpnn_nn_query(const icpnn_tree* tree, const float* xyz, int64_t n, int32_t* idx,
                   float* dist2, uint32_t flags, void* stream);

/* icpnn_voxel_downsample -- the voxel-grid filter of page section 4.3 (run
 * before the tree is built): one output point per occupied voxel of side
 * voxel_size, the centroid of the points in it.
 *   Voxel of a point: (floor(x / v), floor(y / v), floor(z / v)) with
 *   float32 division (the grid is anchored at the coordinate origin); the
 *   centroid sums its points in input order in double and rounds the mean
 *   to float32; output voxels are ordered by (ix, iy, iz); points with a
 *   non-finite coordinate are dropped.  The result is exact: it equals any
 *   implementation of that definition bit for bit.
 *   xyz        n x 3 float32, device or host.
 *   out_xyz    capacity n x 3 float32, device or host.
 *   out_n      host: number of voxels written.
 * Synchronises `stream`.  Errors: INVALID_ARG (voxel_size <= 0 or not
 * finite, a voxel index beyond 2^40), CUDA, NO_MEMORY. */
int icpnn_voxel_downsample(const float* xyz, int64_t n, float voxel_size, float* out_xyz, int64_t* out_n,
                           void* stream);

/* ------------------------------------------------------------------ ICP --
 * Moments of one correspondence pass (page sections 2.1, 3.3, 4.4): the
 * original source points s_i whose transformed image R s_i + t has a nearest
 * target point q_i within the maximum distance are "accepted";
 *   mu_src = mean of accepted s_i, mu_tgt = mean of their q_i,
 *   H[3a+b] = sum (s_a - mu_src_a)(q_b - mu_tgt_b)  (row-major 3x3),
 *   sum_d2 = sum of accepted dist2, mse = sum_d2 / n_accepted (NaN if none).
 * n_nonfinite counts source points with a NaN/Inf coordinate (never
 * accepted). */
typedef struct icpnn_moments {
    int64_t n_accepted;
    int64_t n_nonfinite;
    double mu_src[3];
    double mu_tgt[3];
    double H[9];
    double sum_d2;
    double mse;
} icpnn_moments;

/* One row per iteration of icp_align. */
typedef struct icpnn_iter_record {
    int32_t iter;        /* 0-based */
    int32_t flags;       /* reserved, 0 */
    int64_t n_accepted;  /* pairs accepted by the distance test in this pass */
    int64_t n_inliers;   /* pairs the final solve used (= n_accepted without
                            ICPNN_RESIDUAL_REJECT) */
    double mse;          /* mean squared distance of the accepted pairs */
    double sigma2;       /* mean squared residual under the first solve (residual
                            rejection only, else 0) */
    double T[16];        /* row-major transform this pass used (before the solve) */
    float kernel_ms;     /* device time of the pass (with ICPNN_TRACE_TIMING), else 0:
                            on the persistent kernel's clock from the command
                            reaching the GPU to the result published; CUDA events
                            around the launch otherwise, where a one-at-a-time
                            pre-launched pass's time includes its wait for the
                            transform (ICPNN_NO_PRELAUNCH times the kernel alone) */
    float residual_ms;   /* with ICPNN_TRACE_TIMING and ICPNN_RESIDUAL_REJECT in the
                            persistent kernel: device time of the iteration's two
                            residual passes (command seen to the second's result
                            published), else 0 */
} icpnn_iter_record;

/* icpnn_icp_step -- one fused correspondence pass under a given float32
 * transform (R row-major 3x3, t): transform the original source points,
 * search, reject pairs with double(dist2) > max_corr_dist^2, reduce.
 *   src          n x 3 float32 source points (device, or host: copied in).
 *   R, t         host float32 arrays (9 and 3).
 *   max_corr_dist  <= 0 or infinite: no rejection.
 *   idx, dist2   optional (NULL) per-point outputs in the source's order, as in
 *                icpnn_nn_query (device or host memory).
 *   out          host moments.
 * Synchronises `stream`.  Errors: INVALID_ARG, NOT_UPLOADED, CUDA,
 * NO_MEMORY, NONFINITE (when n_nonfinite > 0; `out` is still filled). */
int icpnn_icp_step(const icpnn_tree* tree, const float* src, int64_t n, const float* R,
                   const float* t, double max_corr_dist, int32_t* idx, float* dist2,
                   icpnn_moments* out, void* stream);

/* icpnn_kabsch -- the host solve of page section 2.1 from a moments record:
 * H = U S V^T by a one-sided Jacobi SVD in double, R = V diag(1, 1,
 * sign det(V U^T)) U^T (reflection guard), t = mu_tgt - R mu_src.  Writes
 * the 4x4 row-major transform to T.  Errors: INVALID_ARG, DEGENERATE
 * (n_accepted < 3 or sigma_2 <= 1e-12 sigma_1).  Host only. */
int icpnn_kabsch(const icpnn_moments* m, double* T);

/* icpnn_icp_align -- the whole registration (page section 3.3 loop, section
 * 4.6 stopping rule):
 *   T_0 = init_T (row-major 4x4, NULL = identity);
 *   for k = 0 .. max_iter-1: pass under float32(T_k) (icpnn_icp_step), fail
 *   with DEGENERATE if fewer than 3 pairs are accepted, mse_k, T_{k+1} =
 *   icpnn_kabsch; stop after the solve once k >= 2 and
 *   |mse_{k-1} - mse_k| < eps and |mse_{k-2} - mse_{k-1}| < eps.
 *   With ICPNN_RESIDUAL_REJECT (page section 4.4) each iteration's first
 *   solve T' is followed by: e_i^2 = squared residual of every accepted pair
 *   under float32(T') (the search's float arithmetic), sigma^2 = mean e_i^2,
 *   keep the pairs with double(e_i^2) <= 9 sigma^2, T_{k+1} = solve over the
 *   kept pairs (DEGENERATE if fewer than 3 remain).  The stopping rule still
 *   uses mse_k of the correspondence pass.
 *   Then one more pass (no solve) under the returned transform.
 *   Pass launches: by default the whole registration is one persistent
 *   kernel on `stream` (a cooperative launch: every block resident at once),
 *   which stages the top of the tree once and keeps each SM's cache of the
 *   tree from one pass to the next; between passes its blocks wait on the GPU
 *   for the transform the host writes to pinned memory after each solve.
 *   With ICPNN_RESIDUAL_REJECT it also runs each iteration's two residual
 *   passes, handing the threshold from one to the other on the GPU.  With
 *   ICPNN_NO_PERSISTENT (or when the grid cannot be resident at once) each
 *   pass is instead queued while the previous one runs and waits the same
 *   way (not with ICPNN_RESIDUAL_REJECT); with ICPNN_NO_PRELAUNCH every pass
 *   is an ordinary launch after its solve.  Every wait is bounded (50 ms): a
 *   pass that runs out (a profiler that serialises launches, a host thread
 *   descheduled that long) is run again as an ordinary launch and so is the
 *   rest of the registration.  Results are bit-identical in every mode.
 *   With ICPNN_TRACE_TIMING, kernel_ms is the pass's time on the persistent
 *   kernel's clock (command seen to result published), or CUDA events around
 *   the pass otherwise (0 for passes run after a fallback).
 *   src          n_src x 3 float32 (device, or host: copied in once).
 *   max_iter     >= 1.  eps >= 0 (0: run max_iter iterations).
 *   out_T        host double[16]: the last solved transform (target ~ T src).
 *   final_mse    host: mse of the extra pass (NaN if nothing accepted).
 *   iters        host: number of solves performed.
 *   final_n_accepted  optional host int64: pairs accepted by the extra pass.
 *                final_n_accepted / n_src is the overlap ratio of page
 *                section 6, which advises a warning when it falls below
 *                ICPNN_OVERLAP_WARN_RATIO after registration (a symptom of
 *                a wrong stopping rule or a failed registration).  With no
 *                maximum distance every finite point is accepted and the
 *                ratio is 1.
 *   trace        optional host array of trace_cap records (one per
 *                iteration, up to trace_cap).
 *   flags        ICPNN_TRACE_TIMING | ICPNN_RESIDUAL_REJECT |
 *                ICPNN_NO_PRELAUNCH | ICPNN_NO_PERSISTENT, or 0.
 * Synchronises `stream` once per iteration; scratch comes from the
 * stream-ordered allocator and is returned before the call ends.
 * Errors: INVALID_ARG, NOT_UPLOADED, CUDA, NO_MEMORY, NONFINITE, DEGENERATE. */
#define ICPNN_OVERLAP_WARN_RATIO 0.8
int icpnn_icp_align(const icpnn_tree* target, const float* src, int64_t n_src, int32_t max_iter,
                    double eps, double max_corr_dist, const double* init_T, double* out_T,
                    double* final_mse, int32_t* iters, int64_t* final_n_accepted,
                    icpnn_iter_record* trace, int32_t trace_cap, uint32_t flags, void* stream);

/* icpnn_icp_align_batch -- register n_frames sources against one resident
 * target (page section 3.4: several frames in flight so that one frame's
 * queries overlap another frame's result transfer and solve).  Each frame is
 * an icpnn_icp_align run by a library worker thread on a stream of its own,
 * with up to max_concurrent frames in flight (<= 0: 4); frames are handed out
 * in order as workers free up.  Every frame's result is bit-identical to a
 * single-frame icpnn_icp_align of it.
 *   srcs, n_src   n_frames source pointers (n x 3 float32, device or host)
 *                 and point counts.
 *   init_T        NULL or n_frames row-major 4x4 initial transforms.
 *   out_T, final_mse, iters, status   per-frame outputs (host arrays of
 *                 16*n_frames, n_frames, n_frames, n_frames); status[f] is
 *                 frame f's icpnn_status.
 *   final_n_accepted  optional host int64[n_frames]: as for icpnn_icp_align.
 *   flags         ICPNN_RESIDUAL_REJECT | ICPNN_NO_PRELAUNCH, or 0; with more
 *                 than one frame in flight passes are never pre-launched
 *                 (a waiting pass would hold SM slots other frames can use).
 *   stream        the frames start after work already enqueued on it; all
 *                 their work is complete when the call returns.
 * Returns ICPNN_OK if every frame succeeded, else the first failing frame's
 * status (icpnn_last_error names the frame).  The caller's current device must
 * be the tree's.  Errors: INVALID_ARG, NOT_UPLOADED, CUDA, NO_MEMORY,
 * NONFINITE, DEGENERATE. */
int icpnn_icp_align_batch(const icpnn_tree* target, int32_t n_frames, const float* const* srcs,
                          const int64_t* n_src, int32_t max_iter, double eps, double max_corr_dist,
                          const double* init_T, double* out_T, double* final_mse, int32_t* iters,
                          int64_t* final_n_accepted, int32_t* status, uint32_t flags,
                          int32_t max_concurrent, void* stream);

/* ------------------------------------------------------ no allocation --
 * icpnn_icp_step_noalloc -- the fused correspondence pass of icpnn_icp_step
 * for callers that cannot allocate device memory: code embedded in a host
 * application or framework that owns all device memory and hands out only
 * its own buffers, processes whose device memory is fully reserved by
 * another allocator, and real-time loops that cannot afford cudaMalloc /
 * cudaFree (cudaFree waits for the whole device) or an allocation failure
 * in the middle of a frame.  The paper has no counterpart: it is an
 * integration aid, not part of the method.
 *   The result is the same pass: same per-point idx/dist2 (bit for bit) and
 *   the same moments up to float rounding order (the points are visited in
 *   the caller's order, not Morton order, so partial sums associate
 *   differently).
 *   src          n x 3 float32, memory of the current device (host pointers
 *                and other GPUs' memory are rejected).
 *   n            1 .. ICPNN_NOALLOC_MAX_POINTS; larger n is rejected with
 *                ICPNN_ERR_INVALID_ARG (one thread per point; one partial
 *                record per 256 points must fit the scratch array).
 *   R, t, max_corr_dist, out   as for icpnn_icp_step.
 *   idx, dist2   both NULL or both buffers of n entries in the current
 *                device's memory.
 * Scratch: a fixed file-scope device array of ICPNN_NOALLOC_MAX_POINTS/256
 * partial records plus a few words (about 576 KB), created when the library
 * is loaded and held by every GPU that loads it until the process exits.  No
 * call allocates or frees memory, host or device (the 18-double result is
 * copied into the caller's `out` through a stack buffer).
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for later calls.
 * Sharing: every call on a device uses the same array, and each call leaves
 * its contents behind (the counter that must start at zero is cleared at the
 * start of every call).  Calls that overlap on the GPU -- concurrent streams
 * or threads on one device -- race on the array and give wrong results;
 * serialise them.  The call synchronises `stream`.
 * Errors: INVALID_ARG, NOT_UPLOADED, CUDA, NONFINITE (as icpnn_icp_step). */
#define ICPNN_NOALLOC_MAX_POINTS 1048576
int icpnn_icp_step_noalloc(const icpnn_tree* tree, const float* src, int64_t n, const float* R,
                           const float* t, double max_corr_dist, int32_t* idx, float* dist2,
                           icpnn_moments* out, void* stream);

/* ----------------------------------------------------------------- misc -- */

/* Message for the calling thread's most recent failed call ("" if none). */
const char* icpnn_last_error(void);

/* Number of kernels this library has launched in this process (all threads). */
int64_t icpnn_launch_count(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t icpnn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ICPNN_H */
