/*
 * oracle.c -- the plain, slow, obviously correct CPU definition of the
 * gradient all-reduce and its halves.  TEST INFRASTRUCTURE ONLY: it is
 * built and called by the tests, by the smoke check and by the benchmark's
 * CPU-baseline leg, never by the product path.  It shares no code with the
 * CUDA library.
 *
 * What is computed, and where the pages fix it:
 *
 *  - All-reduce: every participant contributes a tensor of the same size and
 *    every participant receives the elementwise sum, or the mean
 *    ("Distributed Training", computervisiononline.com, "Data parallelism and
 *    all-reduce"; "Lecture 8 -- Parallelism", rd.me/cs336/lec8, Part 1 s.2,
 *    dist.all_reduce with SUM or AVG; Burn's ReduceOperation {Sum, Mean},
 *    pgsm.cn/news/420861, "Distributed tensor operations").
 *  - Reduce-scatter: the reduced tensor is split and each participant keeps
 *    one part (cielbird.github.io/blog/burn-distributed, "Collective
 *    operations"; Lecture 8, Part 1 s.2, dist.reduce_scatter).
 *  - All-gather: every participant receives the concatenation of all parts
 *    (Lecture 8, Part 1 s.2, dist.all_gather).
 *  - Broadcast: one participant's tensor is copied to all others
 *    (burn-distributed, "Collective operations"; Lecture 8, dist.broadcast).
 *  - Buckets: gradients are packed into buckets of about 25 MB, filled in the
 *    reverse order of the parameters, one collective per bucket
 *    ("Distributed Training", "Data parallelism and all-reduce").
 *  - The optimizer step follows the all-reduce (Lecture 8, Part 2 s.1,
 *    steps 3-4); momentum is the optimizer state the pages name
 *    ("Distributed Training", the paragraph on parameter averaging).
 *
 * Readings where the pages leave a step open (each listed in the design notes):
 *  - summation order: ascending rank, sequential fp32 adds, the accumulator
 *    seeded with rank 0's value (a sum of one term is that term, so -0.0
 *    survives); the pages only warn that the order changes the last digits
 *    ("Distributed Training", "Equivalence");
 *  - Mean = the fp32 sum, then one correctly rounded fp32 division by P;
 *  - bf16 inputs widen exactly to fp32; the fp32 result is rounded once to
 *    bf16, to nearest with ties to even (FP32 accumulation, as in mixed
 *    precision training);
 *  - reduce-scatter shards are contiguous: rank r keeps [r*N/P, (r+1)*N/P),
 *    N % P == 0; all-gather concatenates in rank order;
 *  - SGD with momentum mu and learning rate lr, dampening 0, on the fp32
 *    reduced gradient g, each product and sum rounded separately:
 *    v = fl(fl(mu*v) + g);  w = fl(w - fl(lr*v)).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * fp32 arithmetic is IEEE binary32 with round-to-nearest-even; no FMA
 * contraction, no flush-to-zero.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_SUM = 0, OR_MEAN = 1 };
enum { OR_OK = 0, OR_BAD = 1 };

/* bf16 -> fp32: a bf16 value is the upper half of an fp32 bit pattern. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * fp32 -> bf16, round to nearest, ties to even (IEEE 754 rounding of the
 * 24-bit significand to 8 bits).  Adding 0x7FFF plus the lowest kept bit and
 * truncating rounds up exactly when the dropped half is above one half, or
 * equal to one half with an odd kept part; a carry out of the significand
 * moves into the exponent, which also turns the largest finite values that
 * round up into infinity.  NaN keeps its sign and upper payload and is made
 * quiet.
 */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* The same cast over an array (for tests that probe many values). */
void oracle_f32_to_bf16_array(const float *x, uint16_t *y, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        y[i] = oracle_f32_to_bf16(x[i]);
}

static size_t elem_size(int dtype) { return dtype == OR_BF16 ? 2 : 4; }

static float load(const void *p, size_t i, int dtype)
{
    if (dtype == OR_BF16)
        return oracle_bf16_to_f32(((const uint16_t *)p)[i]);
    return ((const float *)p)[i];
}

static void store(void *p, size_t i, int dtype, float v)
{
    if (dtype == OR_BF16)
        ((uint16_t *)p)[i] = oracle_f32_to_bf16(v);
    else
        ((float *)p)[i] = v;
}

/* One reduced element: x_0[i] + x_1[i] + ... + x_{P-1}[i], left to right in
 * fp32, then divided by P for Mean. */
static float reduce_one(int P, const void *const *x, size_t i, int dtype, int op)
{
    float acc = load(x[0], i, dtype);
    for (int r = 1; r < P; ++r)
        acc = acc + load(x[r], i, dtype);
    if (op == OR_MEAN)
        acc = acc / (float)P;
    return acc;
}

static int bad_args(int P, int dtype, int op)
{
    return P < 1 || (dtype != OR_F32 && dtype != OR_BF16) || (op != OR_SUM && op != OR_MEAN);
}

/* All-reduce: recv[r][i] = reduce(send[0..P-1][i]) for every rank r.
 * recv[r] may be send[r] (in place). */
int oracle_all_reduce(int P, const void *const *send, void *const *recv, size_t n,
                      int dtype, int op)
{
    if (bad_args(P, dtype, op))
        return OR_BAD;
    for (size_t i = 0; i < n; ++i) {
        float y = reduce_one(P, send, i, dtype, op);
        for (int r = 0; r < P; ++r)
            store(recv[r], i, dtype, y);
    }
    return OR_OK;
}

/* Reduce-scatter: rank r receives shard r of the reduced tensor,
 * recv[r][j] = reduce(send[.][r*n/P + j]) for j < n/P. */
int oracle_reduce_scatter(int P, const void *const *send, void *const *recv, size_t n,
                          int dtype, int op)
{
    if (bad_args(P, dtype, op) || n % (size_t)P != 0)
        return OR_BAD;
    size_t shard = n / (size_t)P;
    for (int r = 0; r < P; ++r)
        for (size_t j = 0; j < shard; ++j)
            store(recv[r], j, dtype, reduce_one(P, send, (size_t)r * shard + j, dtype, op));
    return OR_OK;
}

/* All-gather: recv[r] = send[0] ++ send[1] ++ ... ++ send[P-1], each send[s]
 * holding n/P elements.  A bit copy. */
int oracle_all_gather(int P, const void *const *send, void *const *recv, size_t n, int dtype)
{
    if (P < 1 || (dtype != OR_F32 && dtype != OR_BF16) || n % (size_t)P != 0)
        return OR_BAD;
    size_t bytes = n / (size_t)P * elem_size(dtype);
    for (int r = 0; r < P; ++r)
        for (int s = 0; s < P; ++s) {
            char *dst = (char *)recv[r] + (size_t)s * bytes;
            if (dst != (const char *)send[s])
                memcpy(dst, send[s], bytes);
        }
    return OR_OK;
}

/* Broadcast: buf[r] = buf[root] for every rank r.  A bit copy. */
int oracle_broadcast(int P, void *const *buf, size_t n, int dtype, int root)
{
    if (P < 1 || root < 0 || root >= P || (dtype != OR_F32 && dtype != OR_BF16))
        return OR_BAD;
    for (int r = 0; r < P; ++r)
        if (r != root)
            memcpy(buf[r], buf[root], n * elem_size(dtype));
    return OR_OK;
}

/*
 * Bucketed all-reduce with an optional SGD-momentum step.  ptrs holds the
 * replicas tensor-major (ptrs[t*P + r]); numel[t] is tensor t's length.
 * Without SGD each tensor is all-reduced in place.  With SGD (master and
 * momentum non-NULL), the reduced fp32 gradient g drives
 *     v <- fl(fl(momentum * v) + g),   w <- fl(w - fl(lr * v))
 * on tensor t's fp32 master[t] and momentum[t]; the replicas then receive
 * the reduced gradient only when write_back is non-zero.
 */
int oracle_bucket_all_reduce(int P, int ntensors, void *const *ptrs, const uint64_t *numel,
                             int dtype, int op, float lr, float momentum,
                             float *const *master, float *const *momentum_buf, int write_back)
{
    if (bad_args(P, dtype, op) || ntensors < 0)
        return OR_BAD;
    int sgd = master != NULL && momentum_buf != NULL;
    for (int t = 0; t < ntensors; ++t) {
        void *const *x = ptrs + (size_t)t * (size_t)P;
        for (size_t i = 0; i < numel[t]; ++i) {
            float g = reduce_one(P, (const void *const *)x, i, dtype, op);
            if (sgd) {
                float *v = momentum_buf[t], *w = master[t];
                float mv = momentum * v[i];
                v[i] = mv + g;
                float step = lr * v[i];
                w[i] = w[i] - step;
            }
            if (!sgd || write_back)
                for (int r = 0; r < P; ++r)
                    store(x[r], i, dtype, g);
        }
    }
    return OR_OK;
}

/*
 * Bucket assignment: walk the tensors from the last registered to the first
 * and add each to the open bucket; a tensor that would take a non-empty
 * bucket past cap_bytes opens a new bucket first (so a tensor larger than
 * the cap sits alone).  bucket_of[t] receives tensor t's bucket; buckets are
 * numbered in the order they fill.  Returns the number of buckets, or -1.
 */
int oracle_bucket_plan(int ntensors, const uint64_t *nbytes, uint64_t cap_bytes, int *bucket_of)
{
    if (ntensors < 0 || cap_bytes == 0)
        return -1;
    int b = -1;
    uint64_t fill = 0;
    for (int t = ntensors - 1; t >= 0; --t) {
        if (b < 0 || (fill > 0 && fill + nbytes[t] > cap_bytes)) {
            ++b;
            fill = 0;
        }
        bucket_of[t] = b;
        fill += nbytes[t];
    }
    return b + 1;
}

/*
 * Gradient accumulation with DDP's no_sync ("Distributed Training",
 * "Gradient accumulation": a device processes a batch as micro-batches in
 * sequence and adds their gradients before one optimizer step, each
 * micro-batch's loss divided by the number of micro-batches M; DDP's
 * no_sync() skips the all-reduce until the last micro-batch).
 *
 * oracle_bucket_accumulate (a micro-batch before the last, no all-reduce):
 * for every tensor t, rank r and element i, with s = fl(scale * g_r[i]),
 *     acc_r[i] = first ? s : fl(acc_r[i] + s)
 * acc is tensor-major like ptrs (acc[t*P + r], fp32, numel[t] elements).
 *
 * oracle_bucket_all_reduce_accumulated (the last micro-batch): every rank's
 * total a_r[i] = first ? s : fl(acc_r[i] + s) is all-reduced exactly as
 * oracle_bucket_all_reduce reduces the gradients themselves (rank order,
 * Mean / P, optional SGD, result stored to every gradient replica unless
 * SGD runs without write-back).  acc is not modified.
 */
int oracle_bucket_accumulate(int P, int ntensors, void *const *ptrs, const uint64_t *numel,
                             int dtype, float *const *acc, float scale, int first)
{
    if (P < 1 || ntensors < 0 || (dtype != OR_F32 && dtype != OR_BF16))
        return OR_BAD;
    for (int t = 0; t < ntensors; ++t)
        for (int r = 0; r < P; ++r) {
            const void *g = ptrs[(size_t)t * (size_t)P + (size_t)r];
            float *a = acc[(size_t)t * (size_t)P + (size_t)r];
            for (size_t i = 0; i < numel[t]; ++i) {
                float s = scale * load(g, i, dtype);
                a[i] = first ? s : a[i] + s;
            }
        }
    return OR_OK;
}

int oracle_bucket_all_reduce_accumulated(int P, int ntensors, void *const *ptrs,
                                         const uint64_t *numel, int dtype, int op,
                                         float *const *acc, float scale, int first, float lr,
                                         float momentum, float *const *master,
                                         float *const *momentum_buf, int write_back)
{
    enum { MAXP = 64 };
    if (bad_args(P, dtype, op) || P > MAXP || ntensors < 0)
        return OR_BAD;
    int sgd = master != NULL && momentum_buf != NULL;
    for (int t = 0; t < ntensors; ++t) {
        void *const *x = ptrs + (size_t)t * (size_t)P;
        float *const *a = acc + (size_t)t * (size_t)P;
        for (size_t i = 0; i < numel[t]; ++i) {
            float total[MAXP];
            for (int r = 0; r < P; ++r) {
                float s = scale * load(x[r], i, dtype);
                total[r] = first ? s : a[r][i] + s;
            }
            float g = total[0];
            for (int r = 1; r < P; ++r)
                g = g + total[r];
            if (op == OR_MEAN)
                g = g / (float)P;
            if (sgd) {
                float *v = momentum_buf[t], *w = master[t];
                float mv = momentum * v[i];
                v[i] = mv + g;
                float step = lr * v[i];
                w[i] = w[i] - step;
            }
            if (!sgd || write_back)
                for (int r = 0; r < P; ++r)
                    store(x[r], i, dtype, g);
        }
    }
    return OR_OK;
}

/*
 * Sharded SGD step, ZeRO stage 1 ("Distributed Training", "Sharded data
 * parallelism: ZeRO and FSDP": the optimizer state is partitioned across the
 * ranks and each rank updates only its partition; the updated parameters
 * then go to all ranks -- ZeroRedundancyOptimizer broadcasts them, FSDP
 * all-gathers the shards).  With s = n / P, rank r owns elements
 * [r*s, (r+1)*s) and holds that part of the fp32 master weights and
 * momentum in w_shard[r], v_shard[r] (s elements each).  Three steps:
 *   1. reduce-scatter: rank r's part of the reduced gradient, g (fp32,
 *      before any rounding) = reduce(grads[.][r*s + j]);
 *   2. the owner's SGD step on its shard: v = fl(fl(mu*v) + g),
 *      w = fl(w - fl(lr*v));
 *   3. all-gather: every rank's params[q][r*s + j] = w, rounded to dtype.
 */
int oracle_sharded_sgd_step(int P, const void *const *grads, void *const *params,
                            float *const *w_shard, float *const *v_shard, size_t n, int dtype,
                            int op, float lr, float momentum)
{
    if (bad_args(P, dtype, op) || n % (size_t)P != 0)
        return OR_BAD;
    size_t s = n / (size_t)P;
    for (int r = 0; r < P; ++r)
        for (size_t j = 0; j < s; ++j) {
            size_t i = (size_t)r * s + j;
            float g = reduce_one(P, grads, i, dtype, op);
            float *v = v_shard[r], *w = w_shard[r];
            float mv = momentum * v[j];
            v[j] = mv + g;
            float step = lr * v[j];
            w[j] = w[j] - step;
            for (int q = 0; q < P; ++q)
                store(params[q], i, dtype, w[j]);
        }
    return OR_OK;
}

/*
 * Synchronized batch-normalization statistics ("Distributed Training",
 * "Synchronized batch normalization": the per-shard statistics are pooled
 * over the ranks so every rank normalizes with the statistics of the whole
 * batch; the example pools the per-shard sums and sums of squares with an
 * all-reduce, mean = s1 / n, var = s2 / n - mean^2, the biased variance of
 * training mode, and normalizes with sqrt(var + eps)).
 * sum[r][c], sqsum[r][c]: rank r's fp32 sums of x and x*x over its values of
 * channel c; count[r]: rank r's number of values per channel.  In fp64,
 * ranks added in order 0..P-1:
 *     n = count[0] + ... + count[P-1],  s1 = sum[0][c] + ... , s2 = ...,
 *     mean = s1 / n,  var = s2 / n - mean * mean,  invstd = 1 / sqrt(var + eps);
 * every rank receives mean and invstd rounded to fp32.
 */
int oracle_syncbn_stats(int P, const float *const *sum, const float *const *sqsum,
                        const uint64_t *count, float *const *mean, float *const *invstd,
                        size_t channels, float eps)
{
    if (P < 1)
        return OR_BAD;
    uint64_t n_total = 0;
    for (int r = 0; r < P; ++r)
        n_total += count[r];
    if (n_total == 0)
        return OR_BAD;
    double n = (double)n_total;
    for (size_t c = 0; c < channels; ++c) {
        double s1 = (double)sum[0][c], s2 = (double)sqsum[0][c];
        for (int r = 1; r < P; ++r) {
            s1 = s1 + (double)sum[r][c];
            s2 = s2 + (double)sqsum[r][c];
        }
        double m = s1 / n;
        double var = s2 / n - m * m;
        double is = 1.0 / sqrt(var + (double)eps);
        for (int r = 0; r < P; ++r) {
            mean[r][c] = (float)m;
            invstd[r][c] = (float)is;
        }
    }
    return OR_OK;
}
