/*
 * gar.h -- C ABI of libgar.so, the GB300 gradient all-reduce library.
 *
 * A device group of P participants (ranks) is P replica buffers resident in
 * the HBM of one GPU.  Each collective is one kernel pass over all P
 * replicas: it reads every participant's tensor and writes the result for
 * every participant.  The calls follow the problem as the pages state it:
 *   - a device group with a default reduction, created before any
 *     collective and alive while the group is in use (Burn's
 *     DistributedContext::init(devices, DistributedConfig{all_reduce_op})
 *     and its Drop; pgsm.cn/news/420861, "Distributed tensor operations" and
 *     "Lifetime and implementation details");
 *   - ReduceOperation Sum or Mean (same page, "Reduction configuration";
 *     "Lecture 8 -- Parallelism", rd.me/cs336/lec8, Part 1 s.2: SUM or AVG);
 *   - the same tensor on every participant, the result returned to each
 *     (same page, all_reduce; Lecture 8, dist.all_reduce);
 *   - results that are asynchronous until synchronised (same page,
 *     CollectiveTensor::resolve): every call enqueues work on the caller's
 *     CUDA stream and returns; the output is valid once that stream has
 *     reached the call (cudaStreamSynchronize, an event, or later work on the
 *     same stream).
 * Because one call takes all P participants at once, the pages' rule that
 * every participant joins the same collectives in a compatible order holds
 * by construction.
 *
 * Numerics (identical to the CPU oracle bit for bit): element i of the
 * result is x_0[i] + x_1[i] + ... + x_{P-1}[i], added left to right in IEEE
 * fp32 starting from x_0[i]; Mean then divides once by P in fp32 (correctly
 * rounded).  bf16 inputs widen exactly to fp32 and the fp32 result is
 * rounded once to bf16 (nearest, ties to even).  A NaN result is a NaN; its
 * payload is not specified.
 *
 * Ownership: the caller owns every buffer and stream.  The library never
 * allocates or frees caller memory; a comm owns one small device status
 * word.  Pointers: device memory (or memory the device can address) on the
 * comm's device, aligned to the element size; 16-byte alignment selects the
 * vectorised path, other alignments run a scalar path with the same
 * results.  Counts are elements per participant; count == 0 is a no-op that
 * inspects no buffer pointer (they may be NULL).
 * Errors: every call validates its arguments on the host before enqueueing
 * anything and returns AR_ERR_INVALID_ARG with nothing enqueued when they
 * are wrong; AR_ERR_CUDA reports a failed CUDA call or launch.
 * Threading: a comm is not thread-safe; calls on one comm must be
 * serialised by the caller.  Calls leave the calling thread's current
 * CUDA device unchanged.
 */
#ifndef GAR_H
#define GAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AR_MAX_RANKS 16

typedef struct ar_comm_s *ar_comm_t;

typedef enum {
    AR_OK = 0,
    AR_ERR_INVALID_ARG = 1, /* bad argument; nothing was enqueued */
    AR_ERR_UNSUPPORTED = 2, /* no sm_103a device, or a feature not built */
    AR_ERR_CUDA = 3,        /* a CUDA runtime call or a kernel launch failed */
    AR_ERR_TIMEOUT = 4,     /* a device-side bounded wait gave up */
    AR_ERR_STATE = 5,       /* a comm used after ar_destroy, or not from ar_init */
    AR_ERR_DEVICE_CHECK = 6 /* a debug build's device-side index check failed */
} ar_status_t;

/* ReduceOperation.  AR_OP_DEFAULT selects the comm's default_op. */
typedef enum { AR_OP_DEFAULT = -1, AR_SUM = 0, AR_MEAN = 1 } ar_op_t;

/* Element types: IEEE binary32, and bfloat16 (the upper half of a binary32). */
typedef enum { AR_F32 = 0, AR_BF16 = 1 } ar_dtype_t;

/* A CUDA stream handle (cudaStream_t); NULL is the legacy default stream. */
typedef void *ar_stream_t;

/*
 * Create a device group of nranks participants (1 <= nranks <= AR_MAX_RANKS)
 * on CUDA device cuda_device, with default reduction default_op (AR_SUM or
 * AR_MEAN).  Cites DistributedContext::init and DistributedConfig
 * (pgsm.cn/news/420861, "Distributed tensor operations").  On success *comm
 * holds the new handle; it allocates a 4-byte device status word.
 * Errors: AR_ERR_INVALID_ARG (null comm, nranks or default_op out of range,
 * no such device), AR_ERR_UNSUPPORTED (the device is not sm_103),
 * AR_ERR_CUDA.
 */
ar_status_t ar_init(ar_comm_t *comm, int nranks, int cuda_device, ar_op_t default_op);

/*
 * Destroy a group (the Drop of DistributedContext, same page, "Lifetime and
 * implementation details").  Waits for the device to finish work that may
 * use the status word, then frees it.  AR_ERR_STATE for a handle that is
 * not live.
 */
ar_status_t ar_destroy(ar_comm_t comm);

/*
 * All-reduce (Lecture 8, Part 1 s.2, dist.all_reduce; "Distributed
 * Training", computervisiononline.com, "Data parallelism and all-reduce").
 * send[r], recv[r] (host arrays of P device pointers): count elements each.
 * recv[r][i] = reduce_op(send[0][i], ..., send[P-1][i]) for every rank r.
 * recv[r] == send[r] is in place; otherwise recv[r] must not overlap any
 * send[q] or recv[q].  recv buffers of different ranks must be disjoint;
 * send buffers may overlap each other (they are only read).
 */
ar_status_t ar_all_reduce(ar_comm_t comm, const void *const *send, void *const *recv,
                          size_t count, ar_dtype_t dtype, ar_op_t op, ar_stream_t stream);

/*
 * Reduce-scatter (Lecture 8, Part 1 s.2, dist.reduce_scatter;
 * burn-distributed, "Collective operations").  count % P == 0; shard
 * s = count / P.  send[r]: count elements; recv[r]: s elements.
 * recv[r][j] = reduce_op(send[.][r*s + j]): rank r keeps the contiguous
 * shard r.  In place iff recv[r] == send[r] + r*s (elements); otherwise
 * recv[r] must not overlap any send or other recv.
 */
ar_status_t ar_reduce_scatter(ar_comm_t comm, const void *const *send, void *const *recv,
                              size_t count, ar_dtype_t dtype, ar_op_t op, ar_stream_t stream);

/*
 * All-gather (Lecture 8, Part 1 s.2, dist.all_gather; "Distributed
 * Training", FSDP paragraphs).  count % P == 0 is the TOTAL length;
 * s = count / P.  send[r]: s elements; recv[r]: count elements.
 * recv[r][q*s + j] = send[q][j], a bit copy in rank order.  In place iff
 * send[r] == recv[r] + r*s; otherwise send and recv must not overlap.
 */
ar_status_t ar_all_gather(ar_comm_t comm, const void *const *send, void *const *recv,
                          size_t count, ar_dtype_t dtype, ar_stream_t stream);

/*
 * Broadcast (Lecture 8, Part 1 s.2, dist.broadcast; burn-distributed,
 * "Collective operations"; DDP's broadcast of rank 0's state, "Distributed
 * Training", "Data parallelism and all-reduce").  buf[r]: count elements;
 * afterwards every buf[r] holds buf[root]'s bytes; buf[root] is only read.
 * The P buffers must be disjoint; 0 <= root < P.
 */
ar_status_t ar_broadcast(ar_comm_t comm, void *const *buf, size_t count, ar_dtype_t dtype,
                         int root, ar_stream_t stream);

/*
 * A gradient bucket: ntensors tensors of one dtype, each with P replicas.
 * dev_ptrs is a HOST array of ntensors*P device pointers, tensor-major
 * (dev_ptrs[t*P + r] is rank r's copy of tensor t); numel is a HOST array of
 * ntensors lengths.  Buckets of about 25 MB, filled in reverse parameter
 * order, one collective per bucket ("Distributed Training", "Data
 * parallelism and all-reduce"); see ar_bucket_plan.
 */
typedef struct {
    int ntensors;
    void *const *dev_ptrs;
    const size_t *numel;
    ar_dtype_t dtype;
} ar_bucket_t;

/*
 * The optimizer step that follows the all-reduce (Lecture 8, Part 2 s.1,
 * step 4, optimizer.step()), as SGD with momentum (dampening 0): for each
 * element, with g the fp32 reduced gradient before any bf16 rounding,
 *     v = fl(fl(momentum * v) + g),   w = fl(w - fl(lr * v)).
 * master[t] and momentum_buf[t] (HOST arrays of ntensors device pointers)
 * are fp32 arrays of numel[t] elements, shared by all replicas (they hold
 * the same values after the all-reduce).  write_back_grads != 0 also stores
 * the reduced gradient (rounded to the bucket dtype) into every replica; 0
 * leaves the gradient replicas untouched.
 */
typedef struct {
    float lr;
    float momentum;
    float *const *master;
    float *const *momentum_buf;
    int write_back_grads;
} ar_sgd_t;

/*
 * Bucketed all-reduce, in place: every tensor of the bucket is all-reduced
 * exactly as ar_all_reduce would (bucketing cannot change values), in one
 * kernel launch for buckets of up to 256 tensors at P <= 8 (128 at P <= 16;
 * larger buckets take one launch per such group).  sgd == NULL: results go
 * to every replica.  sgd != NULL: the fused SGD-momentum step above.  All
 * buffers (replicas, master, momentum) must be pairwise disjoint.
 */
ar_status_t ar_bucket_all_reduce(ar_comm_t comm, const ar_bucket_t *bucket, ar_op_t op,
                                 const ar_sgd_t *sgd, ar_stream_t stream);

/*
 * Gradient accumulation with DDP's no_sync ("Distributed Training",
 * "Gradient accumulation": a batch processed as M micro-batches in sequence,
 * their gradients added before one optimizer step, each micro-batch's loss
 * divided by M; DDP's no_sync() skips the all-reduce until the last
 * micro-batch).  acc is a HOST array of ntensors*P fp32 device pointers,
 * tensor-major like ar_bucket_t.dev_ptrs (acc[t*P + r]: numel[t] elements,
 * rank r's accumulator of tensor t).  scale multiplies every micro-batch
 * gradient (1/M for the mean over M micro-batches; 1 to add them as they
 * are).  first = 1 starts a cycle: the accumulators are overwritten.
 */
typedef struct {
    float *const *acc;
    float scale;
    int first;
} ar_accum_t;

/*
 * A micro-batch before the last, with no all-reduce: per tensor t, rank r
 * and element i, with s = fl(scale * g_r[i]) (the gradient widened to fp32),
 * acc_r[i] = first ? s : fl(acc_r[i] + s).  The gradients are only read.
 * Buffer rules as for ar_bucket_all_reduce, plus: every accumulator is
 * fp32, 4-byte aligned and disjoint from every other buffer.
 */
ar_status_t ar_bucket_accumulate(ar_comm_t comm, const ar_bucket_t *grads, const ar_accum_t *acc,
                                 ar_stream_t stream);

/*
 * The last micro-batch: rank r's total t_r[i] = first ? s : fl(acc_r[i] + s)
 * with s = fl(scale * g_r[i]) is all-reduced exactly as ar_bucket_all_reduce
 * reduces gradients (rank order, Mean / P, the optional fused SGD step), and
 * the result goes to every gradient replica (unless SGD runs without
 * write-back).  The accumulators are only read; the next cycle starts with
 * first = 1.  first = 1 with scale = 1 is exactly ar_bucket_all_reduce.
 */
ar_status_t ar_bucket_all_reduce_accumulated(ar_comm_t comm, const ar_bucket_t *grads,
                                             const ar_accum_t *acc, ar_op_t op,
                                             const ar_sgd_t *sgd, ar_stream_t stream);

/*
 * Sharded SGD step, ZeRO stage 1 ("Distributed Training", "Sharded data
 * parallelism: ZeRO and FSDP": the optimizer state is partitioned over the
 * ranks, each rank updates only its partition, and the updated parameters
 * go to every rank).  count % P == 0, s = count / P.  grads[r], params[r]:
 * count elements of dtype; master_shards[r], momentum_shards[r]: rank r's
 * s fp32 elements of the master weights and momentum, for elements
 * [r*s, (r+1)*s).  One fused pass does the three collectives of the step:
 * reduce-scatter of the gradients (g in fp32, before any rounding, reduced
 * as by ar_all_reduce), the owner's SGD step on its shard
 * (v = fl(fl(momentum*v) + g), w = fl(w - fl(lr*v))), and the all-gather
 * of the updated weights, rounded to dtype, into every params[q].
 * params[r] == grads[r] is in place; otherwise params and grads are
 * disjoint.  The shards are disjoint from everything.  The vectorised path
 * needs every shard to start on a 16-byte boundary: pad the flat unit so
 * that s * sizeof(dtype) is a multiple of 16 (other sizes run the scalar
 * path, with the same results).
 */
ar_status_t ar_sharded_sgd_step(ar_comm_t comm, const void *const *grads, void *const *params,
                                float *const *master_shards, float *const *momentum_shards,
                                size_t count, ar_dtype_t dtype, ar_op_t op, float lr,
                                float momentum, ar_stream_t stream);

/*
 * Synchronized batch-normalization statistics ("Distributed Training",
 * "Synchronized batch normalization": per-shard statistics pooled over the
 * ranks, so every rank normalizes with the statistics of the whole batch;
 * the page's example all-reduces the per-shard sums and sums of squares).
 * sum[r], sqsum[r]: rank r's fp32 per-channel sums of x and of x*x over its
 * shard (channels values each); count: HOST array of P values, rank r's
 * number of values per channel (their total must be > 0 and <= 2^53).
 * For every channel, in fp64 with the ranks added in order 0..P-1:
 *   n = sum of count, s1 = sum over r of sum[r], s2 = likewise,
 *   mean = s1 / n,  var = s2 / n - mean^2 (biased, as in training),
 *   invstd = 1 / sqrt(var + eps);
 * every rank's mean[r], invstd[r] (fp32, channels values) receive them.  A
 * negative var + eps gives NaN.  Outputs must be disjoint from each other
 * and from the inputs.  Latency-bound: one thread per channel.
 */
ar_status_t ar_syncbn_stats(ar_comm_t comm, const float *const *sum, const float *const *sqsum,
                            const uint64_t *count, float *const *mean, float *const *invstd,
                            size_t channels, float eps, ar_stream_t stream);

/*
 * Bucket assignment, host only.  nbytes[t] is tensor t's size in
 * registration order.  Tensors are taken from the last to the first and
 * added to the open bucket; one that would take a non-empty bucket past
 * cap_bytes opens a new bucket first, so a tensor larger than the cap sits
 * alone ("Distributed Training", "Data parallelism and all-reduce": 25 MB
 * buckets, reverse parameter order).  bucket_of[t] receives tensor t's
 * bucket index (buckets numbered in fill order); *nbuckets their number.
 * Errors: AR_ERR_INVALID_ARG for ntensors < 0, cap_bytes == 0, or null
 * outputs (bucket_of may be null when ntensors == 0).
 */
ar_status_t ar_bucket_plan(int ntensors, const size_t *nbytes, size_t cap_bytes,
                           int *bucket_of, int *nbuckets);

/*
 * DDP gradient reducer: the bucketing engine of DDP.  Gradients are packed
 * into buckets of about 25 MB in reverse parameter order and an
 * asynchronous all-reduce is launched on each bucket as soon as all of its
 * gradients are ready, while the backward pass goes on; every rank reduces
 * the buckets in the same order ("Distributed Training", "Data parallelism
 * and all-reduce").  A reducer holds the whole group's gradient set and
 * does per step what ar_bucket_all_reduce does per bucket, with identical
 * results, but validates and plans only once.
 *
 * ar_reducer_create: grads lists EVERY gradient tensor in registration
 * order (the layout of ar_bucket_t); buckets are planned with
 * ar_bucket_plan(cap_bytes); op as for the collectives; sgd NULL, or the
 * fused SGD-momentum step of ar_sgd_t (per-tensor master / momentum).  All
 * buffers are validated here with the rules of ar_bucket_all_reduce and
 * must stay allocated, at the same addresses, while the reducer lives.
 * Creates two communication streams (the device's highest priority) and
 * three events on the comm's device; destroy the reducer before its comm.
 * Not thread-safe.
 */
typedef struct ar_reducer_s *ar_reducer_t;
ar_status_t ar_reducer_create(ar_reducer_t *reducer, ar_comm_t comm, const ar_bucket_t *grads,
                              size_t cap_bytes, ar_op_t op, const ar_sgd_t *sgd);

/*
 * Tensor `tensor` (its P replicas) holds its final gradient of this step
 * once `stream` reaches the call.  When the last tensor of a bucket is
 * marked, that bucket's kernel is launched on a communication stream,
 * ordered after every stream that marked one of its tensors (consecutive
 * buckets alternate between the two streams and may overlap on the GPU).
 * Exception: a call that completes every bucket of the step when every
 * tensor of the step was marked on one stream launches on that stream
 * itself (nothing of the step is left to overlap with; consecutive steps
 * on one stream then chain without events between their kernels).
 * AR_ERR_INVALID_ARG for an index out of range; AR_ERR_STATE for a tensor
 * already marked in this step.
 */
ar_status_t ar_reducer_mark_ready(ar_reducer_t reducer, int tensor, ar_stream_t stream);

/* ar_reducer_mark_ready for tensors[0], tensors[1], ... (one call for a
 * group of gradients that become final together).  All or nothing: when an
 * index is out of range (AR_ERR_INVALID_ARG), already marked or listed
 * twice (AR_ERR_STATE), no tensor is marked.  The buckets the call
 * completes are launched at its end, in completion order; consecutive ones
 * whose combined segment table fits one launch (<= 256 tensors, <= 2048
 * replica pointers) share a single kernel launch, with the same results
 * and every bucket's completion (ar_reducer_wait_bucket) recorded after
 * it.  Launched on the communication streams, or on `stream` itself as
 * for ar_reducer_mark_ready. */
ar_status_t ar_reducer_mark_ready_many(ar_reducer_t reducer, const int *tensors, int n,
                                       ar_stream_t stream);

/*
 * End of the step: launches every bucket not launched yet (its unmarked
 * tensors are taken as ready on `stream`; combined launches and the
 * choice of stream as in ar_reducer_mark_ready_many), makes `stream` wait
 * for all the step's buckets (no host blocking), and clears the marks for
 * the next step.
 */
ar_status_t ar_reducer_finalize(ar_reducer_t reducer, ar_stream_t stream);

/*
 * Makes `stream` wait (no host blocking) for bucket `bucket` of the current
 * step -- e.g. to copy that bucket's results out while later buckets are
 * still being produced (DDP's per-bucket completion).  For a bucket
 * launched on its marking stream (see ar_reducer_mark_ready) the wait
 * covers that stream's work up to this call.  AR_ERR_STATE if the bucket
 * has not been launched in this step; AR_ERR_INVALID_ARG for an index
 * outside 0 .. nbuckets-1 (see ar_reducer_info).
 */
ar_status_t ar_reducer_wait_bucket(ar_reducer_t reducer, int bucket, ar_stream_t stream);

/* New SGD learning rate and momentum for the following launches (a
 * learning-rate schedule); AR_ERR_INVALID_ARG if the reducer has no SGD. */
ar_status_t ar_reducer_set_sgd(ar_reducer_t reducer, float lr, float momentum);

/* Number of buckets and, if bucket_of is not NULL, each tensor's bucket. */
ar_status_t ar_reducer_info(ar_reducer_t reducer, int *nbuckets, int *bucket_of);

/* *launches = kernel launches the reducer has issued since it was created
 * (one per launch table of a bucket launched alone, one per combined
 * launch; buckets whose tensors are all empty launch nothing).  Host-side
 * count: no device synchronisation.  AR_ERR_INVALID_ARG for a null output. */
ar_status_t ar_reducer_launches(ar_reducer_t reducer, uint64_t *launches);

/* Waits for the reducer's streams, then frees it.  AR_ERR_STATE if not live. */
ar_status_t ar_reducer_destroy(ar_reducer_t reducer);

/*
 * Sticky device-side status of a comm: AR_ERR_DEVICE_CHECK once a kernel of
 * a debug build (compiled with GAR_DEBUG=1) found an index outside the
 * buffers its launch describes (the access is skipped, nothing traps);
 * AR_ERR_TIMEOUT once a kernel's bounded wait has given up; AR_ERR_CUDA for
 * a sticky CUDA error on the device; else AR_OK.  Synchronises the device
 * (it reads the status word).
 */
ar_status_t ar_get_async_error(ar_comm_t comm);

/*
 * Failure-detection self-test.  Enqueues one warp that waits, with the
 * bounded mbarrier wait of the bulk-copy pipeline, on a barrier that
 * nothing ever arrives at; after timeout_ms (1..2000) the wait gives up and
 * records the timeout in the comm's status word, exactly as a stalled
 * pipeline stage would.  The GPU context stays usable; afterwards
 * ar_get_async_error(comm) returns AR_ERR_TIMEOUT for this comm (the status
 * is sticky: destroy the comm).  The pages have no counterpart: DDP's
 * collectives simply block until every rank joins ("Distributed Training",
 * "Data parallelism and all-reduce").
 */
ar_status_t ar_selftest_wait_timeout(ar_comm_t comm, unsigned timeout_ms, ar_stream_t stream);

/*
 * All-reduce that allocates nothing -- for callers that may not allocate
 * device memory themselves and so cannot call ar_init (it allocates the
 * comm's status word): plugins whose host framework owns every device
 * allocation through its own pool, services that reserve all memory at
 * start-up and forbid allocations while serving (cudaMalloc can stall the
 * device), code running under a hard memory cap.  The pages have no
 * counterpart for this entry point.
 *
 * Same operation, arguments and checks as ar_all_reduce, for nranks
 * participants on the CALLER'S CURRENT CUDA device, with op AR_SUM or
 * AR_MEAN (no comm, so no default op); results are identical bit for bit.
 * It always runs the bulk-copy pipelined kernel.  The caller passes inputs
 * and outputs; the kernel's scratch -- one 4-byte status word set when a
 * bounded wait gives up -- lives in a static 256-byte device array that
 * every GPU loading the library holds until the process exits.  Every call
 * needs that one word whatever its arguments (a compile-time check keeps
 * it inside the array), so no call can ask for more scratch than the
 * array holds.  The call allocates no memory: no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * The first call on a device sets that device up (checks it is sm_103 and
 * looks up the array's device address in the device's context).  The
 * address is kept for the rest of the process: do not call this entry
 * point on a device after cudaDeviceReset has destroyed the context it was
 * set up in.  Every call clears the status word on `stream` before its
 * launch.  All calls on a device share the one array, so calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race on
 * it; calls on one stream are ordered and do not.  The status word has no
 * comm to be read through: a wait that gave up (after 2 s) leaves the
 * outputs incomplete without an error code here; callers who need that
 * report use ar_init and ar_get_async_error.
 * Errors: AR_ERR_INVALID_ARG as for ar_all_reduce; AR_ERR_UNSUPPORTED when
 * the current device is not sm_103 (or has index >= 64); AR_ERR_CUDA.
 */
ar_status_t ar_all_reduce_noalloc(int nranks, const void *const *send, void *const *recv,
                                  size_t count, ar_dtype_t dtype, ar_op_t op, ar_stream_t stream);

/* A static, human-readable name for a status code. */
const char *ar_status_string(ar_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GAR_H */
