/*
 * psgd.h -- C ABI of the GB300 PowerSGD compression step (libpsgd.so).
 *
 * What it computes (PowerSGD review page, "PowerSGD: Practical Low-Rank
 * Gradient Compression for Distributed Optimization", section 提案手法 /
 * proposed method):  for every layer whose gradient is an n x m matrix and
 * for W data-parallel workers w,
 *     M_w   = G_w + E_w                       error feedback      (bullet 3)
 *     P     = sum_w M_w Q                     first all-reduce    (bullets 1, 2)
 *     Phat  = Gram-Schmidt(P)                 orthonormal columns (bullet 1)
 *     Q_w   = M_w^T Phat                      power-iteration step
 *     Qbar  = (1/W) sum_w Q_w                 second all-reduce   (bullet 2)
 *     U     = Phat Qbar^T                     decompression       (bullet 5)
 *     E_w  <- M_w - Phat Q_w^T                new error           (bullet 3)
 *     Q    <- Qbar                            warm start of the next step (bullet 1)
 * with P in R^{n x r} and Q in R^{m x r}, r small (bullet 4).  A 1-D tensor
 * (a bias or a batch-norm vector) is averaged over the workers and sent whole.
 * The W workers live on one GPU: each "all-reduce" is a sum over the worker
 * axis inside the kernels.  All values are float32.
 *
 * Readings of points the page leaves open:
 *   - P is a sum over workers, Qbar a mean, so U approximates the mean gradient;
 *   - E_w uses the worker's own Q_w;
 *   - Q starts as N(0,1) draws: splitmix64 keyed by (seed, layer) + Box-Muller
 *     (see psgd_create);
 *   - a column of P whose Gram-Schmidt remainder is zero gives a zero column.
 *
 * Layout of a packed gradient buffer (one per worker, float32, device memory):
 * every layer l sits at element offset psgd_layer_info(..).offset, 16-byte
 * aligned; a matrix layer is row-major n x ld with ld = m rounded up to a
 * multiple of 4 (the ld - m padding columns are ignored on input and written
 * as 0 on output); a vector layer is n contiguous floats (the floats after it,
 * up to the next layer, are neither read nor written).  The decompressed
 * update (out_update) uses the same layout.
 *
 * Ownership: the caller owns the gradient buffers and out_update.  The library
 * owns the error state, P, Q and all scratch, allocated by psgd_create and
 * freed by psgd_destroy; it never frees caller memory.
 *
 * Errors: every call returns a psgd_status; nothing throws across the ABI.
 * psgd_last_error() gives a message for the calling thread.  psgd_step is
 * asynchronous on the context's stream (no host synchronisation); a CUDA
 * error raised while it runs is reported by the next synchronising call
 * (psgd_sync or any psgd_get_*), after which the context only answers
 * PSGD_ERR_STATE until destroyed.
 *
 * Launches: a PowerSGD step is one kernel per phase (project, orthonormalise,
 * back-project, decompress; at r >= 8 a fifth forms the second Cholesky-QR
 * pass's Phat rows), each a grid of independent tiles over all layers
 * launched as a programmatic dependent of the one before; none waits on
 * another CTA.  At r >= 16 the project phase's products run on the tensor
 * cores (tcgen05, error-compensated TF32); a wait on them that runs out is
 * reported as PSGD_ERR_TIMEOUT.
 *
 * One-pass project (options.one_pass; psgd_step at padded rank 1, 2 or 4,
 * every worker in this process): the project phase runs on clusters of
 * 8 CTAs that together hold whole rows of a layer and exchange the row
 * block's partial P rows through distributed shared memory, so each block's
 * P rows are complete on chip; the CTAs then accumulate Y_w = M_w^T P from
 * the M rows they just wrote (read back from L2).  Since Phat = P R^-1 after
 * one Cholesky-QR pass, Q_w = M_w^T Phat = Y_w R^-1, and the back-project
 * forms Q_w from Y without reading M from memory again -- for each layer
 * whose P has kappa_F(R) <= 128 (the rounding of Y R^-1 grows with kappa);
 * other layers' back-project reads M as in the two-pass form.  The kernels
 * per step are the same four.  psgd_layer_flags tells which form a layer
 * took.  A layer set whose widest layer needs more than 8 CTAs per row at
 * the rank's thread limit (W x ceil(m / 4) > 8 x 256 x 16 / RP) keeps the
 * two-pass form.
 *
 * With options.fused (padded rank 1, 2 or 4, one process) a step
 * is instead ONE launch whose CTAs take the tiles of all four phases from one
 * queue in dependency order; a tile whose inputs another CTA is still
 * producing waits for a flag.  Every such wait is bounded (options.wait_ms,
 * 2 s by default): one that runs out abandons the step, and the next
 * synchronising call answers PSGD_ERR_TIMEOUT (the context is then unusable,
 * the CUDA context is not harmed).
 *
 * Thread safety: a context must not be used from two host threads at once.
 * Two contexts are independent and may run concurrently on different streams.
 */
#ifndef PSGD_H_
#define PSGD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct psgd_ctx psgd_ctx;

typedef enum {
  PSGD_OK = 0,
  PSGD_ERR_INVALID = -1,  /* bad argument (null / misaligned pointer, bad size, rank) */
  PSGD_ERR_OOM = -2,      /* device or pinned-host allocation failed */
  PSGD_ERR_CUDA = -3,     /* a CUDA runtime call failed (message in psgd_last_error) */
  PSGD_ERR_TIMEOUT = -4,  /* a fused step waited past options.wait_ms and was abandoned */
  PSGD_ERR_STATE = -5     /* the context hit an earlier error and is unusable */
} psgd_status;

/* Cumulative counters of a context (exact integers). */
typedef struct {
  int64_t steps;                        /* psgd_step calls enqueued */
  int64_t floats_sent;                  /* per worker, summed over steps: sum (n+m) r + vector lengths */
  int64_t floats_uncompressed;          /* per worker, summed over steps: sum n m + vector lengths */
  int64_t floats_sent_per_step;         /* per worker, one step */
  int64_t floats_uncompressed_per_step; /* per worker, one step */
  int64_t matrix_elements;              /* per worker: sum over matrix layers of n*m */
  int64_t vector_elements;              /* per worker: sum over vector layers of n */
  int64_t buffer_elements;              /* floats in one packed gradient buffer (with padding) */
  int64_t tiles[4];                     /* CTAs of the project, orthonormalise, back-project, decompress kernels */
  int32_t kernel_rank;                  /* rank the kernels were compiled for (r rounded up to 1,2,4,8,16,32) */
  int32_t launches_per_step;            /* kernels one psgd_step enqueues (with an update) */
  int32_t tile_rows[3];                 /* rows per tile: project, back-project (least), decompress */
  int32_t fused_step;                   /* 1: each step is one fused launch (see the header comment) */
  int64_t message_floats;               /* floats psgd_step_host writes to msg_host */
  int32_t one_pass_project;             /* 1: psgd_step runs the one-pass project (see "Launches") */
  int32_t reserved_;
} psgd_stats;

/* Optional knobs of psgd_create_ex (zero-initialise, then set what you need). */
typedef struct {
  int32_t timing;       /* 1: time every phase of every step with CUDA events (psgd_get_phase_times) */
  int32_t project_rows; /* rows per project tile (0: chosen so the grid holds several waves of CTAs) */
  int32_t unbiased;     /* 1: the unbiased rank-r variant (see below) instead of PowerSGD */
  int32_t compressor;   /* PSGD_POWERSGD (0) or PSGD_RTOPK (1): rTop-k sparsification (see below) */
  int32_t rtopk_top_div;    /* rTop-k: the top set of a layer of d entries has ceil(d / top_div) */
  int32_t rtopk_sample_div; /* rTop-k: k = ceil(r / sample_div) of them are sent */
  int32_t fused;        /* 1: each step is ONE launch over a queue of every phase's tiles (PowerSGD at
                           r <= 4 in one process; see "Launches" above); 0: one kernel per phase */
  int32_t wait_ms;      /* fused step: longest wait of a tile for its inputs (0: 2000 ms) */
  int32_t queue_lag_kb; /* fused step: bytes of other tiles between a layer's phases in the
                           queue, in KiB (0: about what the resident CTAs hold in flight) */
  int32_t test_stall;   /* tests of the timeout path only: k > 0 never raises the first flag
                           of matrix layer k - 1, so its later tiles wait until wait_ms */
  int32_t total_workers; /* workers over all processes when this context's num_workers are one
                            process's share (the split step below); 0: num_workers */
  int32_t one_pass;     /* 1: the one-pass project where it applies (see "Launches");
                           0: the back-project reads M again (two passes over M) */
} psgd_options;

enum { PSGD_POWERSGD = 0, PSGD_RTOPK = 1 };

/*
 * The unbiased rank-r variant (options.unbiased = 1).  The PowerSGD review
 * page (main findings, bullet 4) sets PowerSGD's biased, error-fed compressor
 * against an unbiased rank-r one without defining it; the reading taken is
 * the random-projection estimate.  Every step draws a fresh Q (m x r, N(0,1))
 * from a seed all workers share -- the draw of psgd_create with the seed
 * replaced by the splitmix64 output of seed + (t + 1) * 0x9E3779B97F4A7C15 for
 * step t (the t-th psgd_step of the context, from 0) -- and computes
 *     P = sum_w G_w Q   (the one all-reduce: only P is sent, n r floats)
 *     U = P Q^T / (W r) (unbiased: E[Q Q^T] = r I)
 * with no error feedback, no warm start and no orthonormalisation.  In this
 * variant psgd_get_PQ returns P and the step's Q, psgd_get_error returns
 * zeros, and psgd_get_Qw and psgd_set_state answer PSGD_ERR_INVALID.
 */

/*
 * rTop-k sparsification (options.compressor = PSGD_RTOPK), the second
 * compressor behind this ABI (rTop-k review page, "rTop-k: A Statistical
 * Estimation Approach to Distributed SGD", proposed method, bullet 3: a
 * random subset of the top magnitude entries).  Per worker w and matrix
 * layer (d = n m entries, flat row-major index i), with error feedback:
 *     M_w = G_w + E_w                                  (float32)
 *     T   = the r = ceil(d / top_div) entries with the largest (|M_w|, -i)
 *     K   = the k = ceil(r / sample_div) members of T with the smallest
 *           (upper 32 bits of splitmix64(key + (i + 1) * 0x9E3779B97F4A7C15), i),
 *           key = splitmix64_mix(s + (w * 65536 + layer + 1) * 0x9E3779B97F4A7C15),
 *           s = the step seed of the unbiased variant
 *     E_w <- M_w with K zeroed; worker w sends K's indices and values
 *     U   = (sum_w S_w) / W, summed in worker order in float32
 * 1-D tensors are averaged.  Layers must have fewer than 2^31 entries;
 * top_div, sample_div >= 1.  psgd_get_error gives E_w, psgd_get_sparse the
 * message; psgd_get_PQ, psgd_get_Qw, psgd_set_state, psgd_step_momentum and
 * the unbiased option answer PSGD_ERR_INVALID.  psgd_step_host's message is,
 * per matrix layer and per worker in order, the k indices (int32 bits in
 * float slots) then the k values.
 */

/*
 * Create a context for num_layers layers.  Layer l is an n[l] x m[l] matrix,
 * or a vector of length n[l] when m[l] == 0.  rank in [1, 32]; rank <= min(n, m)
 * for every matrix; 1 <= num_workers <= 64.  The error buffers start at zero
 * and each matrix layer's Q at N(0,1) draws from (seed, layer) (see the header
 * comment).  cuda_stream (a cudaStream_t, may be NULL for the legacy default
 * stream) is where every call of this context enqueues its work.  The current
 * CUDA device at the time of the call is the context's device.
 */
int psgd_create(psgd_ctx** out, int num_layers, const int64_t* n, const int64_t* m,
                int rank, int num_workers, uint64_t seed, void* cuda_stream);
int psgd_create_ex(psgd_ctx** out, int num_layers, const int64_t* n, const int64_t* m,
                   int rank, int num_workers, uint64_t seed, void* cuda_stream,
                   const psgd_options* options);
void psgd_destroy(psgd_ctx* ctx);

/* Change the stream later calls enqueue on. */
int psgd_set_stream(psgd_ctx* ctx, void* cuda_stream);

/*
 * One PowerSGD step (every row of the header comment, all layers) on the
 * context's stream.  grad_ptrs: host array of num_workers DEVICE pointers, each
 * to a packed gradient buffer (16-byte aligned) that stays valid until the step
 * has run.  out_update: device packed buffer that receives U for matrix layers
 * and the worker mean for vector layers, or NULL to skip both.  Asynchronous.
 */
int psgd_step(psgd_ctx* ctx, const float* const* grad_ptrs, float* out_update);

/*
 * One step followed by the optimiser update it drives (PowerSGD review page,
 * proposed method, bullet 5: the decompressed update feeds momentum SGD,
 * "EF-SGD with momentum").  The page gives no formula; the reading taken is
 * heavy-ball momentum with a Nesterov-style step, element-wise on every
 * layer (U = Phat Qbar^T for a matrix, the worker mean for a vector):
 *     momentum <- beta * momentum + U
 *     params   <- params - lr * (U + momentum)
 * params and momentum: device packed buffers (the gradient layout, 16-byte
 * aligned), read and written in place by the decompress kernel; their row
 * padding is left as it is.  out_update: as in psgd_step (may be NULL: the
 * update then never goes to memory).  lr and beta must be finite.
 * Asynchronous like psgd_step.
 */
int psgd_step_momentum(psgd_ctx* ctx, const float* const* grad_ptrs, float* params, float* momentum,
                       float lr, float beta, float* out_update);

/*
 * The same step fed from HOST memory.  A worker's packed buffer grad_host[w]
 * in pinned (page-locked, mapped) host memory is read in place by the
 * kernels over the CPU-GPU link; any other host buffer is first copied into a
 * device staging buffer owned by the context (allocated on first use).  Then
 * psgd_step runs, and the compressed message of every matrix layer (Phat
 * then Qbar, each row-major, layers in order: sum (n+m) r floats; P alone in
 * the unbiased variant) is copied into msg_host and, when update_host is not
 * NULL, the packed update into it.  Waits for the copies before returning.
 */
int psgd_step_host(psgd_ctx* ctx, const float* const* grad_host, float* msg_host, float* update_host);

/*
 * The split step: one PowerSGD step whose workers are spread over several
 * processes (one per GPU, the page's deployment: main findings, bullets 1
 * and 6 -- P and Q summed by all-reduce, NCCL or GLOO).  Each process's
 * context holds its own num_workers workers and knows the total
 * (options.total_workers); the caller runs the two all-reduces (sum) between
 * the three calls, on buffers it owns (device memory, float32):
 *
 *   psgd_step_begin(ctx, grads, p_out)  error add, P = sum over this
 *       process's workers of M_w Q  ->  p_out (p_floats: every matrix
 *       layer's n x r block, row-major, layers in order)
 *   -- all-reduce(sum) p_out over the processes into p_sum --
 *   psgd_step_mid(ctx, p_sum, q_out)   Gram-Schmidt of the summed P
 *       (Cholesky-QR2), Q_w = M_w^T Phat for this process's workers, and
 *       (1 / total_workers) sum over them of Q_w  ->  q_out (q_floats: every
 *       matrix layer's m x r block, then every vector layer's n floats of
 *       (1 / total_workers) sum of this process's gradients)
 *   -- all-reduce(sum) q_out into q_sum: Qbar and the vector means --
 *   psgd_step_end(ctx, q_sum, out_update)  Qbar <- q_sum (the next warm
 *       start), U = Phat Qbar^T and the vector means into out_update (may
 *       be NULL)
 *
 * p_floats and q_floats come from psgd_exchange_sizes; they are what one
 * process sends per step ((n + m) r per matrix, vectors whole, as
 * psgd_count_sent).  The all-reduced P is bitwise the same on every process,
 * so every process forms the same Phat.  grads must stay valid until
 * psgd_step_end; p_sum may be p_out and q_sum may be q_out (in-place
 * all-reduce).  Asynchronous on the context's stream; the caller orders its
 * collectives after the enqueued work (same stream, or an event).  The
 * calls must come in the order begin, mid, end (else PSGD_ERR_INVALID, and
 * nothing is enqueued).  psgd_step answers PSGD_ERR_INVALID on a context
 * whose total_workers exceeds num_workers.  PowerSGD only (not the unbiased
 * variant or rTop-k); a context with total_workers == num_workers may use
 * either form, and the split step with the identity as all-reduce gives
 * psgd_step's results.
 */
int psgd_exchange_sizes(const psgd_ctx* ctx, int64_t* p_floats, int64_t* q_floats);
int psgd_step_begin(psgd_ctx* ctx, const float* const* grad_ptrs, float* p_out);
int psgd_step_mid(psgd_ctx* ctx, const float* p_sum, float* q_out);
int psgd_step_end(psgd_ctx* ctx, const float* q_sum, float* out_update);

/* Wait for the context's stream and report a device-side error, if any. */
int psgd_sync(psgd_ctx* ctx);

/*
 * Read results of the last step of layer l (a matrix layer).  Each destination
 * may be host or device memory (or NULL to skip it); the call waits for the
 * copy.  P: n x r row-major (Phat, orthonormal columns).  Q: m x r row-major
 * (Qbar, also the warm start of the next step).
 */
int psgd_get_PQ(psgd_ctx* ctx, int layer, float* P, float* Q);
/*
 * rTop-k: the message of worker w for matrix layer l in the last step --
 * *count (= k) flat indices (ascending, row-major over n x m) into idx and
 * their values into val (host or device memory, either may be NULL).
 */
int psgd_get_sparse(psgd_ctx* ctx, int layer, int worker, int32_t* idx, float* val, int64_t* count);
/* Q_w = M_w^T Phat of worker w in the last step: m x r row-major. */
int psgd_get_Qw(psgd_ctx* ctx, int layer, int worker, float* Q);
/* Error buffer E_w of layer l: dense n x m row-major (host or device memory). */
int psgd_get_error(psgd_ctx* ctx, int layer, int worker, float* E);
/*
 * Overwrite the state of layer l: Q (m x r row-major, the next step's warm
 * start) and, when E is not NULL, E[w] (dense n x m row-major) for every worker;
 * E == NULL sets the errors to zero.  Host or device memory.  With
 * psgd_get_PQ/psgd_get_error this checkpoints and restores a run bit-exactly
 * at r <= 8.  At r >= 16 the project phase rebuilds E on the tensor cores
 * (TF32 products with error compensation, ~2^-21 relative) while
 * psgd_get_error uses float32 multiply-adds, so a restored run agrees with an
 * uninterrupted one to that rounding, not bit for bit.
 */
int psgd_set_state(psgd_ctx* ctx, int layer, const float* Q, const float* const* E);

int psgd_get_stats(const psgd_ctx* ctx, psgd_stats* out);

/*
 * Device time of each phase, in milliseconds, averaged over the steps since
 * the previous call (the last 256 at most): project, orthonormalise,
 * back-project, decompress (ms[4]); for a fused step (stats.fused_step) ms[0]
 * is the whole launch and the other slots are 0; under rTop-k the four slots are its
 * kernels: the pass forming M, the pass listing the top-set candidates, the
 * per-problem selection tail, and the message / error / update writes.
 * Needs options.timing = 1; waits for the stream.  Each timed step records
 * five CUDA events on the stream.
 */
int psgd_get_phase_times(psgd_ctx* ctx, float* ms);

/*
 * Turn the per-phase events on (on != 0) or off for the following steps,
 * whatever options.timing said at creation.  The phase kernels are launched
 * as programmatic dependents of the kernel before them, so each one's CTAs
 * are resident when its predecessor ends; an event recorded between two
 * phases orders them strictly again, so timed steps show each phase alone
 * and untimed steps run with the launches overlapped.
 */
int psgd_set_timing(psgd_ctx* ctx, int on);

/*
 * How the last step treated matrix layer l (the stream is synchronised
 * first): bit 0 of *flags set when one Cholesky-QR pass left Phat
 * orthonormal to working precision (no second pass), bit 1 set when the
 * back-project formed Q_w = (M_w^T P) R^-1 from the one-pass project's
 * partials instead of reading M again (see "Launches").  0 before the first
 * step.  PSGD_ERR_INVALID for a vector layer or a NULL argument.
 */
int psgd_layer_flags(psgd_ctx* ctx, int layer, int32_t* flags);

/* Placement of layer l in a packed buffer: element offset, n, m, row stride. */
int psgd_layer_info(const psgd_ctx* ctx, int layer, int64_t* offset, int64_t* n, int64_t* m,
                    int64_t* ld);

/*
 * psgd_step_noalloc -- one step of ONE matrix layer that allocates nothing.
 *
 * The method itself has no such call; it exists for callers that cannot let
 * a library allocate device memory: a framework that sizes one arena for all
 * of its device memory at start-up (a library cudaMalloc would sit outside
 * the arena and may fail once the arena owns the GPU), or a training loop
 * that must not call cudaMalloc/cudaFree between steps because those calls
 * can synchronise the whole device.  psgd_create allocates the state and
 * scratch of a context; this call takes the state from the caller and keeps
 * its scratch in one fixed device array of PSGD_NOALLOC_SCRATCH_BYTES that is
 * part of the library's device image.  Neither it nor anything it calls
 * allocates memory (host or device).
 *
 * The arithmetic is the step of the header comment for one n x m layer and
 * W = num_workers workers, run by the same kernels and tiling as psgd_step on
 * a one-layer context, so both give the same results.
 *
 * Arguments (all device pointers 16-byte aligned, float32, row-major,
 * ld = m rounded up to a multiple of 4, r = rank):
 *   rank        1, 2, 4, 8, 16 or 32, and <= min(n, m);  1 <= num_workers <= 64
 *   grad_ptrs   host array of W device pointers, each an n x ld gradient
 *               (the ld - m padding columns are ignored)
 *   B           device, W x n x ld, caller-owned error state:
 *                 has_prev == 0: B_w is the error E_w to add (zeros at the
 *                                start); Phat and Qw are not read;
 *                 has_prev != 0: B_w, Phat and Qw are what the previous call
 *                                left, and E_w = B_w - Phat Qw_w^T.
 *               On return B_w holds M_w, so the new error is B_w - Phat Qw_w^T.
 *   Phat        device, n x r: out, the orthonormal P (state for the next call)
 *   Qbar        device, ld x r: in, the warm-start Q (rows m..ld-1 must be
 *               zero); out, Qbar = mean_w Q_w (the next call's warm start;
 *               padding rows stay zero)
 *   Qw          device, W x ld x r: out, Q_w of every worker (state)
 *   out_update  device, n x ld: out, U = Phat Qbar^T (padding columns 0), or NULL
 *   has_prev    0 on the first call of a run, 1 after that (see B)
 *   cuda_stream where the work is enqueued (a cudaStream_t, NULL = legacy default)
 * Asynchronous: returns after enqueueing (five kernel launches, four without
 * out_update); a device error shows at the caller's next synchronisation.
 *
 * Limits and errors: PSGD_ERR_INVALID, with nothing enqueued, for a bad
 * argument or a layer whose scratch would exceed PSGD_NOALLOC_SCRATCH_BYTES
 * (8 MiB; the bulk is W x (row tiles, at most 16) x ld x r x 4 bytes of
 * partial Q_w plus (row blocks) x ld x 32 x r bytes of partial P rows, the
 * tile counts chosen by occupancy as for a context: the largest ResNet-18
 * layer, 512 x 4608 at r = 2 with 4 workers, fits, an 8192 x 8192 layer at
 * r = 4 with 8 workers does not -- use a context for those);
 * PSGD_ERR_CUDA when a CUDA call fails.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and sets the kernels' shared-memory limits; make that
 * first call before any stream capture.  Later calls only enqueue work.  The
 * address and the limits are kept for the life of the process: after a
 * cudaDeviceReset on a device that has seen a call, this entry point must not
 * be called again on it (the kept address would belong to the old context).
 *
 * Concurrency: every call on a device uses the same scratch array.  Two calls
 * whose work overlaps on the device (different streams, or host threads,
 * without ordering between them) race on it and give wrong results; order
 * them on one stream or with events.  The counters in the scratch are cleared
 * by every call itself before its kernels run.
 */
#define PSGD_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int psgd_step_noalloc(int64_t n, int64_t m, int rank, int num_workers,
                      const float* const* grad_ptrs, float* B, float* Phat, float* Qbar,
                      float* Qw, float* out_update, int has_prev, void* cuda_stream);

/*
 * Host-only helpers (no GPU needed).  psgd_plan_layout fills offset[l] and
 * ld[l] (0 for vectors) of the packed layout and *total (floats per buffer).
 * psgd_count_sent gives the floats one worker sends per step with and without
 * compression: (n + m) r per matrix against n m, vectors whole either way.
 */
int psgd_plan_layout(int num_layers, const int64_t* n, const int64_t* m, int64_t* offset,
                     int64_t* ld, int64_t* total);
int psgd_count_sent(int num_layers, const int64_t* n, const int64_t* m, int rank,
                    int64_t* compressed, int64_t* uncompressed);

/*
 * The one-pass project's plan for a layer set (host only, no GPU), for
 * `clusters` resident clusters of 8 CTAs: per matrix layer (counting matrix
 * layers only) 4 int32 in layer_plan -- cw (CTAs across a row), yfc (float4
 * columns per CTA), yr (rows per block), nys (partial slots); and in tiles,
 * 4 int32 each, `clusters` header tiles (0, first segment, segments, 0)
 * followed by the segments (matrix index, first block, end block, slot).
 * With tiles == NULL only *count (header tiles + segments) is set.  Padded
 * rank 1, 2 or 4; PSGD_ERR_INVALID when a layer does not fit the one-pass
 * project (see "Launches").  For checking the plan: every block of every
 * layer belongs to exactly one segment, and the runs are of about equal work.
 */
int psgd_plan_one_pass(int num_layers, const int64_t* n, const int64_t* m, int rank, int num_workers,
                       int clusters, int32_t* layer_plan, int32_t* tiles, int64_t* count);

/*
 * The fused step's queue for a layer set (host only, no GPU): the items a
 * context with these layers would run, in order, 4 int32 each -- (phase << 24
 * | matrix index, a, b, c) with phase 0 project (a = row block, b = segment),
 * 1 orthonormalise (a = row chunk), 2 back-project (a = row tile, b =
 * segment, c = worker), 3 decompress (a = row block, b = segment; c = 1 marks
 * a vector layer's chunk a, its index counting vector layers only).  The
 * matrix index counts matrix layers only.  project_rows: rows per project
 * tile (0: the kernels' maximum); lag_bytes: as options.queue_lag_kb, in
 * bytes.  With items == NULL only *count is set.  For checking the queue's
 * order: every tile comes after the tiles whose results it reads.
 */
int psgd_plan_queue(int num_layers, const int64_t* n, const int64_t* m, int rank, int num_workers,
                    int project_rows, int64_t lag_bytes, int with_update, int32_t* items,
                    int64_t* count);

const char* psgd_last_error(void);
const char* psgd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PSGD_H_ */
