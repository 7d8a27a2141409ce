/*
 * CPU oracle for KD-tree ICP registration.  TEST INFRASTRUCTURE ONLY: it is
 * compiled and called by the tests, by the smoke check and by the CPU-baseline
 * leg of the benchmark, never by the library.  It shares no code with the CUDA
 * path.  Plain, slow, obviously correct C; build with
 *     gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared
 * (no -ffast-math: every float operation below must round on its own, and
 * gcc contracts a*b+c into an FMA on aarch64 unless told not to).
 *
 * Source: "Implementing ICP with CUDA-KDTree" (pwwt.cn/news/5235220).
 *
 *   nn    -- exact 1-nearest neighbour, the correspondence step of section
 *            2.1 (t_i = nearest target point of the transformed s_i).  The
 *            distance is the leaf-loop arithmetic of the section 3.2 query
 *            kernel: dx = ref.x - q.x (same for y, z), d2 = dx*dx + dy*dy +
 *            dz*dz, in float32, evaluated left to right.  The result is
 *            *defined* as the lexicographic minimum of (d2, target index):
 *            equal distances resolve to the lowest target index.
 *   tree  -- the KD-tree of sections 2.2, 3.1, 4.2 and 5.2: an index-linked
 *            node array in recursion (pre-)order, root at 0, leaves with
 *            children -1 and a half-open [start, end) range into a leaf index
 *            table.  Split axis = the axis of largest variance (section 4.2),
 *            split at the median (section 2.2), leaf when the node holds at
 *            most leaf_size points (8-16, section 4.1) or sits at the depth
 *            cap (20, section 5.2).  The round-robin rule of section 4.2
 *            (axis = depth mod 3: x, y, z, x, ...) is the alternative split.
 *   search-- the tree search of section 2.2: walk to the near child first,
 *            then visit the far child unless the splitting plane is farther
 *            than the best distance so far.
 *   transform -- p = R*s + t of section 2.1 applied to the original source
 *            coordinates (section 3.3), float32.
 *   pair_dist2 -- squared distance of given pairs (q_i, p_i) with the same
 *            float32 arithmetic as the search: the residual of a pair under a
 *            transform, for the residual rejection of section 4.4.
 *   voxel -- the voxel-grid downsampling of section 4.3 (done before the
 *            tree is built): one point per occupied voxel, the centroid of the
 *            points in it.  Readings: voxel index floor(x / v) per axis in
 *            float32 (the grid is anchored at the coordinate origin); the
 *            centroid sums the voxel's points in input order in double and
 *            rounds the mean to float32; output voxels ordered by
 *            (ix, iy, iz); points with a non-finite coordinate are dropped.
 *
 * Readings where the page is silent or loose (each also listed in the
 * design notes):
 *   - ties in distance go to the lowest target index (the page's strict
 *     d2 < best keeps the first point visited, which depends on the tree);
 *   - the far child is pruned only when fl(delta*delta) > best (strictly), so
 *     an equally distant, lower-indexed point beyond the plane is still found
 *     (the page writes delta*delta < best);
 *   - leaf iff count <= leaf_size; median index m = floor(count/2), left gets
 *     the m smallest points, right the rest, split value = coordinate of the
 *     m-th smallest; "smallest" orders by (coordinate, point index) so the
 *     partition is unique even with repeated coordinates;
 *   - variance is the population variance computed in double; axes whose
 *     variance is within a relative 1e-9 of the largest count as tied and the
 *     lowest such axis wins, so summation order cannot change the choice;
 *   - the transform evaluates p_a = ((R_a0*s_x + R_a1*s_y) + R_a2*s_z) + t_a,
 *     each operation rounded to float32;
 *   - a query with a non-finite coordinate matches nothing: idx -1, d2 NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- distance */

static float orc_dist2(const float *r, float qx, float qy, float qz)
{
    float dx = r[0] - qx;
    float dy = r[1] - qy;
    float dz = r[2] - qz;
    float sx = dx * dx;
    float sy = dy * dy;
    float sz = dz * dz;
    float s = sx + sy;
    return s + sz;
}

/* (d, i) < (bd, bi) lexicographically */
static int orc_better(float d, int32_t i, float bd, int32_t bi)
{
    return d < bd || (d == bd && i < bi);
}

static int orc_finite3(const float *q)
{
    return isfinite(q[0]) && isfinite(q[1]) && isfinite(q[2]);
}

/* ------------------------------------------------------------- brute force */

/* Exact 1-NN of every query among all m reference points (no tree). */
void orc_nn_brute(const float *ref, int64_t m, const float *q, int64_t n,
                  int32_t *out_idx, float *out_d2)
{
    for (int64_t i = 0; i < n; ++i) {
        const float *qi = q + 3 * i;
        if (!orc_finite3(qi)) {
            out_idx[i] = -1;
            out_d2[i] = NAN;
            continue;
        }
        float bd = INFINITY;
        int32_t bi = INT32_MAX;
        for (int64_t j = 0; j < m; ++j) {
            float d = orc_dist2(ref + 3 * j, qi[0], qi[1], qi[2]);
            if (orc_better(d, (int32_t)j, bd, bi)) {
                bd = d;
                bi = (int32_t)j;
            }
        }
        out_idx[i] = (bi == INT32_MAX) ? -1 : bi;
        out_d2[i] = bd;
    }
}

/* -------------------------------------------------------------- transform */

void orc_transform(const float *R, const float *t, const float *s, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) {
        const float *si = s + 3 * i;
        for (int a = 0; a < 3; ++a) {
            float p0 = R[3 * a + 0] * si[0];
            float p1 = R[3 * a + 1] * si[1];
            float p2 = R[3 * a + 2] * si[2];
            float acc = p0 + p1;
            acc = acc + p2;
            acc = acc + t[a];
            out[3 * i + a] = acc;
        }
    }
}

/* ------------------------------------------------------------- residuals */

/* out[i] = d2 between target point q_i and point p_i, in the search's order
 * of operations (dx = q.x - p.x, ...). */
void orc_pair_dist2(const float *q, const float *p, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_dist2(q + 3 * i, p[3 * i], p[3 * i + 1], p[3 * i + 2]);
}

/* ----------------------------------------------------------------- voxel */

typedef struct {
    int64_t k[3];
    int64_t idx;
} orc_vkey;

static int orc_vkey_cmp(const void *pa, const void *pb)
{
    const orc_vkey *a = (const orc_vkey *)pa, *b = (const orc_vkey *)pb;
    for (int d = 0; d < 3; ++d) {
        if (a->k[d] < b->k[d]) return -1;
        if (a->k[d] > b->k[d]) return 1;
    }
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/* out receives up to n centroids (3 floats each); returns the number of
 * occupied voxels, or -1 on bad arguments / allocation failure. */
int64_t orc_voxel_downsample(const float *xyz, int64_t n, float v, float *out)
{
    if (!(v > 0.0f) || n < 0) return -1;
    orc_vkey *keys = (orc_vkey *)malloc((size_t)(n > 0 ? n : 1) * sizeof(orc_vkey));
    if (!keys) return -1;
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i) {
        const float *p = xyz + 3 * i;
        if (!orc_finite3(p)) continue;
        for (int d = 0; d < 3; ++d) keys[m].k[d] = (int64_t)floorf(p[d] / v);
        keys[m].idx = i;
        ++m;
    }
    qsort(keys, (size_t)m, sizeof(orc_vkey), orc_vkey_cmp);
    int64_t nv = 0;
    for (int64_t a = 0; a < m;) {
        int64_t b = a;
        double sum[3] = {0.0, 0.0, 0.0};
        while (b < m && keys[b].k[0] == keys[a].k[0] && keys[b].k[1] == keys[a].k[1] &&
               keys[b].k[2] == keys[a].k[2]) {
            const float *p = xyz + 3 * keys[b].idx;
            sum[0] += p[0];
            sum[1] += p[1];
            sum[2] += p[2];
            ++b;
        }
        const double cnt = (double)(b - a);
        for (int d = 0; d < 3; ++d) out[3 * nv + d] = (float)(sum[d] / cnt);
        ++nv;
        a = b;
    }
    free(keys);
    return nv;
}

/* ------------------------------------------------------------------- tree */

typedef struct {
    float split_val;     /* splitting coordinate (inner nodes) */
    int32_t split_dim;   /* 0 = x, 1 = y, 2 = z (inner nodes) */
    int32_t left_child;  /* -1 for a leaf */
    int32_t right_child; /* -1 for a leaf */
    int32_t start;       /* leaf: first slot in leaf_index */
    int32_t end;         /* leaf: one past the last slot */
} orc_node;

typedef struct {
    int64_t n;
    float *pts;          /* private copy of the reference cloud, n*3 */
    orc_node *nodes;
    int64_t n_nodes, cap;
    int32_t *leaf_index; /* leaf slot -> reference point index */
    int32_t leaf_size, max_depth, depth;
    int32_t round_robin; /* 0: axis of largest variance, 1: depth mod 3 */
} orc_tree;

static int orc_key_less(const float *pts, int dim, int32_t a, int32_t b)
{
    float fa = pts[3 * (int64_t)a + dim];
    float fb = pts[3 * (int64_t)b + dim];
    return fa < fb || (fa == fb && a < b);
}

static void orc_swap(int32_t *a, int32_t *b)
{
    int32_t t = *a;
    *a = *b;
    *b = t;
}

/* Quickselect: afterwards a[k] is the k-th smallest key, a[0..k) are smaller
 * and a(k..n) larger (keys are unique thanks to the index tie-break). */
static void orc_select(const float *pts, int dim, int32_t *a, int64_t n, int64_t k)
{
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        /* median of three as pivot, moved to a[hi] */
        if (orc_key_less(pts, dim, a[mid], a[lo])) orc_swap(&a[mid], &a[lo]);
        if (orc_key_less(pts, dim, a[hi], a[lo])) orc_swap(&a[hi], &a[lo]);
        if (orc_key_less(pts, dim, a[mid], a[hi])) orc_swap(&a[mid], &a[hi]);
        int32_t pivot = a[hi];
        int64_t store = lo;
        for (int64_t i = lo; i < hi; ++i) {
            if (orc_key_less(pts, dim, a[i], pivot)) {
                orc_swap(&a[i], &a[store]);
                ++store;
            }
        }
        orc_swap(&a[store], &a[hi]);
        if (store == k) return;
        if (k < store) hi = store - 1;
        else lo = store + 1;
    }
}

static int orc_split_axis(const float *pts, const int32_t *a, int64_t n)
{
    double var[3];
    for (int d = 0; d < 3; ++d) {
        double sum = 0.0;
        for (int64_t i = 0; i < n; ++i) sum += pts[3 * (int64_t)a[i] + d];
        double mean = sum / (double)n;
        double ss = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            double e = pts[3 * (int64_t)a[i] + d] - mean;
            ss += e * e;
        }
        var[d] = ss / (double)n;
    }
    double vmax = var[0];
    if (var[1] > vmax) vmax = var[1];
    if (var[2] > vmax) vmax = var[2];
    for (int d = 0; d < 3; ++d)
        if (var[d] >= vmax * (1.0 - 1e-9)) return d;
    return 0;
}

static int32_t orc_push_node(orc_tree *t)
{
    if (t->n_nodes == t->cap) {
        int64_t nc = t->cap ? 2 * t->cap : 64;
        orc_node *nn = (orc_node *)realloc(t->nodes, (size_t)nc * sizeof(orc_node));
        if (!nn) return -1;
        t->nodes = nn;
        t->cap = nc;
    }
    memset(&t->nodes[t->n_nodes], 0, sizeof(orc_node));
    return (int32_t)t->n_nodes++;
}

static int orc_build_rec(orc_tree *t, int64_t lo, int64_t hi, int depth, int32_t *out_node)
{
    int32_t me = orc_push_node(t);
    if (me < 0) return -1;
    *out_node = me;
    if (depth > t->depth) t->depth = depth;
    int64_t count = hi - lo;
    if (count <= t->leaf_size || depth >= t->max_depth) {
        orc_node *nd = &t->nodes[me];
        nd->split_val = 0.0f;
        nd->split_dim = -1;
        nd->left_child = -1;
        nd->right_child = -1;
        nd->start = (int32_t)lo;
        nd->end = (int32_t)hi;
        return 0;
    }
    int32_t *a = t->leaf_index + lo;
    int dim = t->round_robin ? depth % 3 : orc_split_axis(t->pts, a, count);
    int64_t m = count / 2;
    orc_select(t->pts, dim, a, count, m);
    float split = t->pts[3 * (int64_t)a[m] + dim];
    int32_t l, r;
    if (orc_build_rec(t, lo, lo + m, depth + 1, &l)) return -1;
    if (orc_build_rec(t, lo + m, hi, depth + 1, &r)) return -1;
    orc_node *nd = &t->nodes[me]; /* realloc may have moved the array */
    nd->split_val = split;
    nd->split_dim = dim;
    nd->left_child = l;
    nd->right_child = r;
    nd->start = (int32_t)lo;
    nd->end = (int32_t)hi;
    return 0;
}

void orc_tree_free(orc_tree *t)
{
    if (!t) return;
    free(t->pts);
    free(t->nodes);
    free(t->leaf_index);
    free(t);
}

/* Returns 0 on success, -1 on bad arguments or non-finite input, -2 on
 * allocation failure. */
int orc_tree_build(const float *pts, int64_t n, int32_t leaf_size, int32_t max_depth,
                   int32_t round_robin, orc_tree **out)
{
    *out = NULL;
    if (!pts || n < 1 || n > INT32_MAX || leaf_size < 1 || max_depth < 0) return -1;
    for (int64_t i = 0; i < 3 * n; ++i)
        if (!isfinite(pts[i])) return -1;
    orc_tree *t = (orc_tree *)calloc(1, sizeof(orc_tree));
    if (!t) return -2;
    t->n = n;
    t->leaf_size = leaf_size;
    t->max_depth = max_depth;
    t->round_robin = round_robin ? 1 : 0;
    t->pts = (float *)malloc((size_t)n * 3 * sizeof(float));
    t->leaf_index = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    if (!t->pts || !t->leaf_index) {
        orc_tree_free(t);
        return -2;
    }
    memcpy(t->pts, pts, (size_t)n * 3 * sizeof(float));
    for (int64_t i = 0; i < n; ++i) t->leaf_index[i] = (int32_t)i;
    int32_t root;
    if (orc_build_rec(t, 0, n, 0, &root)) {
        orc_tree_free(t);
        return -2;
    }
    *out = t;
    return 0;
}

int64_t orc_tree_num_nodes(const orc_tree *t) { return t->n_nodes; }
int32_t orc_tree_depth(const orc_tree *t) { return t->depth; }

void orc_tree_export(const orc_tree *t, float *split_val, int32_t *split_dim, int32_t *left,
                     int32_t *right, int32_t *start, int32_t *end, int32_t *leaf_index)
{
    for (int64_t i = 0; i < t->n_nodes; ++i) {
        split_val[i] = t->nodes[i].split_val;
        split_dim[i] = t->nodes[i].split_dim;
        left[i] = t->nodes[i].left_child;
        right[i] = t->nodes[i].right_child;
        start[i] = t->nodes[i].start;
        end[i] = t->nodes[i].end;
    }
    memcpy(leaf_index, t->leaf_index, (size_t)t->n * sizeof(int32_t));
}

typedef struct {
    float q[3];
    float bd;
    int32_t bi;
    int64_t nodes, points;
} orc_query;

static void orc_search(const orc_tree *t, int32_t node, orc_query *s)
{
    const orc_node *nd = &t->nodes[node];
    s->nodes++;
    if (nd->left_child < 0) {
        for (int32_t k = nd->start; k < nd->end; ++k) {
            int32_t pi = t->leaf_index[k];
            float d = orc_dist2(t->pts + 3 * (int64_t)pi, s->q[0], s->q[1], s->q[2]);
            s->points++;
            if (orc_better(d, pi, s->bd, s->bi)) {
                s->bd = d;
                s->bi = pi;
            }
        }
        return;
    }
    float axis_val = s->q[nd->split_dim];
    float delta = axis_val - nd->split_val;
    int32_t near = (axis_val < nd->split_val) ? nd->left_child : nd->right_child;
    int32_t far = (axis_val < nd->split_val) ? nd->right_child : nd->left_child;
    orc_search(t, near, s);
    float lb = delta * delta;
    if (!(lb > s->bd)) orc_search(t, far, s);
}

/* Exact 1-NN through the tree.  nodes_visited / points_visited (nullable)
 * receive, per query, how many nodes the search entered and how many
 * reference points it measured. */
void orc_tree_nn(const orc_tree *t, const float *q, int64_t n, int32_t *out_idx, float *out_d2,
                 int64_t *nodes_visited, int64_t *points_visited)
{
    for (int64_t i = 0; i < n; ++i) {
        orc_query s;
        s.q[0] = q[3 * i + 0];
        s.q[1] = q[3 * i + 1];
        s.q[2] = q[3 * i + 2];
        s.bd = INFINITY;
        s.bi = INT32_MAX;
        s.nodes = 0;
        s.points = 0;
        if (orc_finite3(s.q)) {
            orc_search(t, 0, &s);
            out_idx[i] = (s.bi == INT32_MAX) ? -1 : s.bi;
            out_d2[i] = s.bd;
        } else {
            out_idx[i] = -1;
            out_d2[i] = NAN;
        }
        if (nodes_visited) nodes_visited[i] = s.nodes;
        if (points_visited) points_visited[i] = s.points;
    }
}
