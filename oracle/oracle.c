/*
 * oracle.c -- CPU oracle for the emulated all-reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this file's library.  The product path (the CUDA
 * library and its Python binding) never includes, links or calls it, and this
 * file includes nothing from the product path.
 *
 * Plain, single-threaded, deliberately slow: one output element at a time,
 * folding the P emulated ranks' inputs in the combination order of the chosen
 * algorithm.  Arithmetic precision: the pages' all-reduce call is made on
 * ncclFloat data ("NCCL and NVSHMEM -- two GPU communication models, side by
 * side", host-code example with ncclAllReduce), so fp32 data is reduced with
 * fp32 (IEEE binary32, round-to-nearest-even) additions; bf16 data is widened
 * to fp32, accumulated in fp32 and rounded once at the end; int32 data uses
 * two's-complement wrap-around.  The file must be compiled with
 * -ffp-contract=off so that no add is fused with the scale multiply.
 *
 * What is computed ("NCCL, NIXL, and Distributed GPU Communication",
 * section "All-reduce"): every rank's buffer is reduced elementwise with
 * sum / min / max and the one result is stored in every rank's receive
 * buffer; DDP then divides by world_size (the optional `scale`).
 *
 * Combination orders (readings of the pages; the pages give no per-element
 * order, so these orders are this project's definition):
 *
 *   RING (also LL): all-reduce = reduce-scatter + all-gather ("NCCL, NIXL,
 *   and Distributed GPU Communication", section "Reduce-scatter"); the ring
 *   takes 2(N-1) steps (lecture_068 page, section 05 "SHARP").  The count is
 *   split into P chunks of L = roundup(ceil(count/P), V) elements, V = 16 bytes
 *   / element size.  Chunk c starts at rank c and visits c+1, c+2, ... so an
 *   element e of chunk c is folded as
 *       acc = x_c[e];  acc = acc (+) x_{(c+k) mod P}[e],  k = 1 .. P-1.
 *
 *   TREE: the double binary tree ("NCCL and NVSHMEM -- two GPU communication
 *   models, side by side", section "double binary tree": two complementary
 *   binary trees run at the same time).  Labels 1..P form an in-order binary
 *   tree: the root is the largest power of two <= P; a label v with
 *   b = lowbit(v) >= 2 has left child v - b/2 and right child v + h, h the
 *   largest of b/2, b/4, ..., 1 with v + h <= P (no right child if none);
 *   odd labels are leaves.  Tree 0 gives rank r the label r+1; tree 1 gives
 *   rank r the label that rank (r-1) mod P has in tree 0, i.e. label v belongs
 *   to rank v mod P.  A node's value is ((own (+) left) (+) right), absent
 *   children skipped.  Elements [0, H) use tree 0 and [H, count) tree 1, with
 *   H = min(count, roundup(ceil(count/2), V)).
 *
 *   Min / max: acc = (x < acc) ? x : acc (min), acc = (x > acc) ? x : acc
 *   (max), in fold order; on ties the earlier operand is kept.
 *
 *   HIERARCHICAL (lecture_068 page, section 06: intra-node reduce-scatter,
 *   inter-node ring all-reduce, intra-node all-gather): P = G groups of Q
 *   ranks, rank r = g*Q + q.  Phase 1 is a ring reduce-scatter inside each
 *   group: the count is cut into Q chunks of L1 = roundup(ceil(count/Q), V)
 *   elements and chunk c1 of group g is folded from local rank c1:
 *       part_g = x_{g,c1} (+) x_{g,c1+1} (+) ... (+) x_{g,c1+Q-1}  (local mod Q).
 *   Phase 2 is a ring all-reduce of chunk c1 across the G groups: the chunk's
 *   len1 elements are cut into G sub-chunks of L2 = roundup(ceil(len1/G), V)
 *   and an element of sub-chunk c2 is folded from group c2:
 *       y = part_{c2} (+) part_{c2+1} (+) ... (+) part_{c2+G-1}   (groups mod G).
 *   Phase 3 only copies.  G = 1 or Q = 1 reduce to the plain ring.
 *
 *   REDUCE-SCATTER ("NCCL, NIXL, and Distributed GPU Communication", section
 *   "Reduce-scatter"): every rank holds P shards of recvcount elements; the
 *   shards are reduced across ranks and rank s receives reduced shard s.
 *   Shard s is folded in the ring order of all-reduce chunk s -- x_s, then
 *   x_{s+1}, ..., x_{s+P-1} -- so that all-reduce = reduce-scatter +
 *   all-gather holds bit for bit whenever the shard length is a whole number
 *   of 16-byte vectors (then the all-reduce's chunks are exactly the shards).
 *
 *   ALL-GATHER (same page, section "All-gather"): rank s contributes
 *   sendcount elements; every rank receives all P contributions back to back,
 *   rank s's at offset s * sendcount.  A copy: no arithmetic.
 *
 *   Epilogue: y = narrow(acc * scale) for floating types when scale != 1,
 *   y = narrow(acc) otherwise; narrow is RNE to bf16, identity for fp32.
 *   scale != 1 is rejected for int32 and for min / max.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_I32 = 2 };
enum { OR_SUM = 0, OR_MIN = 1, OR_MAX = 2 };
enum { OR_ALGO_RING = 1, OR_ALGO_TREE = 2, OR_ALGO_LL = 3 };

#define OR_MAX_RANKS 1024

typedef union {
    float f;
    uint32_t u;
} acc_t;

static size_t elem_size(int dtype) {
    switch (dtype) {
    case OR_F32: return 4;
    case OR_BF16: return 2;
    case OR_I32: return 4;
    default: return 0;
    }
}

/* V: elements per 16-byte vector; chunk boundaries are multiples of V. */
static size_t vec_elems(int dtype) { return 16 / elem_size(dtype); }

static size_t round_up(size_t a, size_t m) { return (a + m - 1) / m * m; }

float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even fp32 -> bf16 (keep the top 16 bits, rounding on the
 * 16 dropped bits; ties go to the even result).  NaN inputs are out of scope
 * for the all-reduce; they are returned as a quiet NaN of the same sign. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
    return (uint16_t)upper;
}

/* Chunk length of the ring split, in elements. */
size_t oracle_ring_chunk_len(size_t count, int P, int dtype) {
    if (P <= 0 || elem_size(dtype) == 0) return 0;
    size_t per = (count + (size_t)P - 1) / (size_t)P;
    return round_up(per, vec_elems(dtype));
}

/* First element folded along tree 1. */
size_t oracle_tree_split(size_t count, int dtype) {
    if (elem_size(dtype) == 0) return 0;
    size_t h = round_up((count + 1) / 2, vec_elems(dtype));
    return h < count ? h : count;
}

static acc_t load_widened(const void* buf, size_t e, int dtype) {
    acc_t a;
    if (dtype == OR_F32) {
        memcpy(&a.f, (const char*)buf + 4 * e, 4);
    } else if (dtype == OR_BF16) {
        uint16_t h;
        memcpy(&h, (const char*)buf + 2 * e, 2);
        a.f = oracle_bf16_to_f32(h);
    } else {
        memcpy(&a.u, (const char*)buf + 4 * e, 4);
    }
    return a;
}

static acc_t combine(acc_t acc, acc_t x, int dtype, int op) {
    if (dtype == OR_I32) {
        int32_t a = (int32_t)acc.u, b = (int32_t)x.u;
        if (op == OR_SUM) acc.u = acc.u + x.u; /* wraps modulo 2^32 */
        else if (op == OR_MIN) acc.u = (uint32_t)((b < a) ? b : a);
        else acc.u = (uint32_t)((b > a) ? b : a);
    } else {
        if (op == OR_SUM) acc.f = acc.f + x.f;
        else if (op == OR_MIN) acc.f = (x.f < acc.f) ? x.f : acc.f;
        else acc.f = (x.f > acc.f) ? x.f : acc.f;
    }
    return acc;
}

static void store_narrowed(void* buf, size_t e, acc_t y, int dtype) {
    if (dtype == OR_F32) {
        memcpy((char*)buf + 4 * e, &y.f, 4);
    } else if (dtype == OR_BF16) {
        uint16_t h = oracle_f32_to_bf16(y.f);
        memcpy((char*)buf + 2 * e, &h, 2);
    } else {
        memcpy((char*)buf + 4 * e, &y.u, 4);
    }
}

/* ---- the two binary trees on labels 1..P ---- */

static int lowbit(int v) { return v & -v; }

static int tree_root(int P) {
    int r = 1;
    while (r * 2 <= P) r *= 2;
    return r;
}

static int tree_left(int v) {
    int b = lowbit(v);
    return b >= 2 ? v - b / 2 : 0;
}

static int tree_right(int v, int P) {
    int b = lowbit(v);
    if (b < 2) return 0;
    for (int h = b / 2; h >= 1; h /= 2)
        if (v + h <= P) return v + h;
    return 0;
}

/* Rank that owns label v in tree t. */
static int tree_owner(int v, int P, int t) { return t == 0 ? v - 1 : v % P; }

static acc_t tree_value(const acc_t* x, int v, int P, int t, int dtype, int op) {
    acc_t acc = x[tree_owner(v, P, t)];
    int l = tree_left(v), r = tree_right(v, P);
    if (l) acc = combine(acc, tree_value(x, l, P, t, dtype, op), dtype, op);
    if (r) acc = combine(acc, tree_value(x, r, P, t, dtype, op), dtype, op);
    return acc;
}

/* Writes tree t's combination expression over x0..x{P-1}: every combine
 * (+) of an accumulated value a with an operand b is printed as "(a+b)". */
static int tree_expr(int v, int P, int t, char* buf, size_t cap, size_t* pos) {
    int l = tree_left(v), r = tree_right(v, P);
    int kids[2] = {l, r};
    for (int i = 0; i < 2; ++i) {
        if (!kids[i]) continue;
        if (*pos + 1 >= cap) return -1;
        buf[(*pos)++] = '(';
    }
    int w = snprintf(buf + *pos, cap - *pos, "x%d", tree_owner(v, P, t));
    if (w < 0 || (size_t)w >= cap - *pos) return -1;
    *pos += (size_t)w;
    for (int i = 0; i < 2; ++i) {
        if (!kids[i]) continue;
        if (*pos + 1 >= cap) return -1;
        buf[(*pos)++] = '+';
        if (tree_expr(kids[i], P, t, buf, cap, pos)) return -1;
        if (*pos + 1 >= cap) return -1;
        buf[(*pos)++] = ')';
    }
    buf[*pos] = 0;
    return 0;
}

/* Expression of tree t (0 or 1) for P ranks; for P = 4, t = 0 it is
 * "(x3+((x1+x0)+x2))". */
int oracle_tree_expr(int P, int t, char* buf, size_t cap) {
    if (P < 1 || P > OR_MAX_RANKS || (t != 0 && t != 1) || cap < 2) return -1;
    size_t pos = 0;
    buf[0] = 0;
    return tree_expr(tree_root(P), P, t, buf, cap, &pos);
}

/* ---- one output element ---- */

static int check_args(int P, int dtype, int op, int algo, float scale) {
    if (P < 1 || P > OR_MAX_RANKS) return -1;
    if (elem_size(dtype) == 0) return -1;
    if (op != OR_SUM && op != OR_MIN && op != OR_MAX) return -1;
    if (algo != OR_ALGO_RING && algo != OR_ALGO_TREE && algo != OR_ALGO_LL) return -1;
    if (scale != 1.0f && (dtype == OR_I32 || op != OR_SUM)) return -2;
    return 0;
}

/* x[r] = rank r's widened input at element e (of `count`). */
static acc_t reduce_element(const acc_t* x, int P, size_t count, size_t e, int dtype,
                            int op, int algo, float scale) {
    acc_t acc;
    if (algo == OR_ALGO_TREE) {
        int t = e < oracle_tree_split(count, dtype) ? 0 : 1;
        acc = tree_value(x, tree_root(P), P, t, dtype, op);
    } else {
        size_t L = oracle_ring_chunk_len(count, P, dtype);
        int c = (int)(e / L);
        acc = x[c];
        for (int k = 1; k < P; ++k) acc = combine(acc, x[(c + k) % P], dtype, op);
    }
    if (dtype != OR_I32 && scale != 1.0f) acc.f = acc.f * scale;
    return acc;
}

/*
 * All-reduce of P buffers of `count` elements each, for output elements
 * [begin, end): recv[r][e] = y[e] for every rank r.  send[r] / recv[r] are host
 * pointers.  Returns 0, -1 for invalid arguments, -2 for a scale the op does
 * not take.
 */
int oracle_allreduce(int P, const void* const* send, void* const* recv, size_t count,
                     size_t begin, size_t end, int dtype, int op, int algo, float scale) {
    int rc = check_args(P, dtype, op, algo, scale);
    if (rc) return rc;
    if (begin > end || end > count) return -1;
    acc_t x[OR_MAX_RANKS];
    for (size_t e = begin; e < end; ++e) {
        for (int r = 0; r < P; ++r) x[r] = load_widened(send[r], e, dtype);
        acc_t y = reduce_element(x, P, count, e, dtype, op, algo, scale);
        for (int r = 0; r < P; ++r) store_narrowed(recv[r], e, y, dtype);
    }
    return 0;
}

/*
 * Sampled form for full-size checks: vals holds P rows of m input values
 * (row r = rank r's inputs at the element indices idx[0..m)), laid out
 * rank-major and contiguous; out[i] receives the reduced, narrowed value of
 * element idx[i] of a `count`-element all-reduce.
 */
int oracle_allreduce_sampled(int P, const void* vals, const size_t* idx, size_t m,
                             size_t count, int dtype, int op, int algo, float scale,
                             void* out) {
    int rc = check_args(P, dtype, op, algo, scale);
    if (rc) return rc;
    acc_t x[OR_MAX_RANKS];
    for (size_t i = 0; i < m; ++i) {
        if (idx[i] >= count) return -1;
        for (int r = 0; r < P; ++r) x[r] = load_widened(vals, (size_t)r * m + i, dtype);
        acc_t y = reduce_element(x, P, count, idx[i], dtype, op, algo, scale);
        store_narrowed(out, i, y, dtype);
    }
    return 0;
}

/*
 * Reduce-scatter of P ranks' buffers of P * recvcount elements: recv[s] (host
 * pointer, recvcount elements) receives reduced shard s.  Returns 0, -1 for
 * invalid arguments, -2 for a scale the op does not take.
 */
int oracle_reduce_scatter(int P, const void* const* send, void* const* recv, size_t recvcount,
                          int dtype, int op, float scale) {
    int rc = check_args(P, dtype, op, OR_ALGO_RING, scale);
    if (rc) return rc;
    acc_t x[OR_MAX_RANKS];
    for (int s = 0; s < P; ++s) {
        for (size_t i = 0; i < recvcount; ++i) {
            size_t e = (size_t)s * recvcount + i;
            for (int r = 0; r < P; ++r) x[r] = load_widened(send[r], e, dtype);
            acc_t acc = x[s];
            for (int k = 1; k < P; ++k) acc = combine(acc, x[(s + k) % P], dtype, op);
            if (dtype != OR_I32 && scale != 1.0f) acc.f = acc.f * scale;
            store_narrowed(recv[s], i, acc, dtype);
        }
    }
    return 0;
}

/*
 * All-gather: recv[r] (P * sendcount elements) receives send[0], ..., send[P-1]
 * back to back, for every rank r.
 */
int oracle_all_gather(int P, const void* const* send, void* const* recv, size_t sendcount,
                      int dtype) {
    if (P < 1 || P > OR_MAX_RANKS || elem_size(dtype) == 0) return -1;
    size_t es = elem_size(dtype);
    for (int r = 0; r < P; ++r)
        for (int s = 0; s < P; ++s)
            for (size_t i = 0; i < sendcount; ++i)
                memcpy((char*)recv[r] + ((size_t)s * sendcount + i) * es,
                       (const char*)send[s] + i * es, es);
    return 0;
}

/* Hierarchical fold of one element (see the header): x[r] = rank r's input. */
static acc_t reduce_element_hier(const acc_t* x, int P, int Q, size_t count, size_t e, int dtype,
                                 int op, float scale) {
    int G = P / Q;
    size_t V = vec_elems(dtype);
    size_t L1 = round_up((count + (size_t)Q - 1) / (size_t)Q, V);
    size_t c1 = e / L1;
    size_t end1 = (c1 + 1) * L1 < count ? (c1 + 1) * L1 : count;
    size_t len1 = end1 - c1 * L1;
    size_t L2 = round_up((len1 + (size_t)G - 1) / (size_t)G, V);
    size_t c2 = (e - c1 * L1) / L2;
    acc_t total = {0};
    for (int j = 0; j < G; ++j) {
        int g = (int)((c2 + (size_t)j) % (size_t)G);
        acc_t part = x[g * Q + (int)(c1 % (size_t)Q)];
        for (int k = 1; k < Q; ++k) part = combine(part, x[g * Q + (int)((c1 + (size_t)k) % (size_t)Q)], dtype, op);
        total = j == 0 ? part : combine(total, part, dtype, op);
    }
    if (dtype != OR_I32 && scale != 1.0f) total.f = total.f * scale;
    return total;
}

/*
 * Hierarchical all-reduce with groups of Q ranks (Q must divide P), output
 * elements [begin, end) to every rank.  Returns 0, -1 invalid, -2 bad scale.
 */
int oracle_allreduce_hier(int P, int Q, const void* const* send, void* const* recv, size_t count,
                          size_t begin, size_t end, int dtype, int op, float scale) {
    int rc = check_args(P, dtype, op, OR_ALGO_RING, scale);
    if (rc) return rc;
    if (Q < 1 || Q > P || P % Q != 0 || begin > end || end > count) return -1;
    acc_t x[OR_MAX_RANKS];
    for (size_t e = begin; e < end; ++e) {
        for (int r = 0; r < P; ++r) x[r] = load_widened(send[r], e, dtype);
        acc_t y = reduce_element_hier(x, P, Q, count, e, dtype, op, scale);
        for (int r = 0; r < P; ++r) store_narrowed(recv[r], e, y, dtype);
    }
    return 0;
}

/* Sampled form of oracle_allreduce_hier (layout as oracle_allreduce_sampled). */
int oracle_allreduce_hier_sampled(int P, int Q, const void* vals, const size_t* idx, size_t m,
                                  size_t count, int dtype, int op, float scale, void* out) {
    int rc = check_args(P, dtype, op, OR_ALGO_RING, scale);
    if (rc) return rc;
    if (Q < 1 || Q > P || P % Q != 0) return -1;
    acc_t x[OR_MAX_RANKS];
    for (size_t i = 0; i < m; ++i) {
        if (idx[i] >= count) return -1;
        for (int r = 0; r < P; ++r) x[r] = load_widened(vals, (size_t)r * m + i, dtype);
        store_narrowed(out, i, reduce_element_hier(x, P, Q, count, idx[i], dtype, op, scale), dtype);
    }
    return 0;
}
