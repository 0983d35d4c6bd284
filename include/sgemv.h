/*
 * sgemv.h -- C ABI of libsgemv: mixed-precision SparseGemv y = W_hat . x on
 * one NVIDIA GB300 (sm_103a).
 *
 * The operation (Dong et al., "Efficient LLM ad generation via model
 * compression and parallel verification", arXiv 2605.11582):
 *   - W is a linear layer's weight, rows x cols (out features x in
 *     features), pruned N:4 along cols -- 2:4 for critical layers, 1:4 for
 *     the rest (section 3.2, "Sparsification"; Figure 1 caption);
 *   - kept weights are quantised to INT4 group-wise with a per-layer group
 *     size (section 1, "Our core idea"; section 3.2, "Adaptive group
 *     quantization"), asymmetric with binary16 scale and zero per group;
 *   - the sparse weight is held in the index-compressed 2bit-CSR form, one
 *     2-bit in-quad position per kept weight (section 1, contribution 1);
 *   - the product is an INT4 weight-only GEMV with mixed sparsity, x and y
 *     in binary16, fp32 accumulation (section 1, contribution 2; section
 *     3.3).
 * Pruning keeps the N largest |w| of each quad (Eq. 3 with equal input
 * norms and no gradient term; ties go to the lower column).  Quantisation
 * per (row, group of g columns) over the kept values S:
 *   lo = min(0, min S), hi = max(0, max S);
 *   s = binary16((hi - lo) / 15) (1.0 if hi == lo; 2^-24 if it rounds to 0);
 *   z = clamp(rint(-lo / s), 0, 15);  q = clamp(rint(w / s) + z, 0, 15);
 *   W_hat = (q - z) * s.  All rounding is to nearest, ties to even.
 *
 * Canonical 2bit-CSR bytes (the import/export format; P = cols*N/4 kept
 * weights per row, kept weight j lies in quad floor(j/N), positions ascend
 * within a quad):
 *   vals : rows x (P/2) bytes, INT4 code of kept j in byte j/2, low nibble
 *          for even j;
 *   idx  : rows x (P/4) bytes, 2-bit position of kept j at bits 2*(j%4) of
 *          byte j/4;
 *   scale, zero : rows x (cols/g) binary16 bit patterns, row-major.
 * On the device the library keeps its own layout of the same information
 * (see sgemv_sizes); export returns the canonical bytes exactly.
 *
 * Conventions for every call:
 *   - the return value is SGEMV_OK (0) or a negative SGEMV_ERR_* code, and
 *     sgemv_last_error() then describes the failure (thread-local text);
 *   - argument errors are detected on the host before anything is launched;
 *   - device pointers (x_dev, y_dev, w_dev) are owned by the caller and must
 *     be on the handle's device; host pointers are owned by the caller and
 *     only read (inputs) or written (outputs) during the call, except for
 *     sgemv_run_host, whose buffers must stay valid until the stream reaches
 *     the end of the call's work;
 *   - a stream argument is a cudaStream_t passed as void*; NULL means the
 *     legacy default stream;
 *   - a handle is not safe for concurrent pack/import/export/destroy.
 *     Products with m = 1 only read the packed weight, so any number of them
 *     may run concurrently on different streams.  Products with m >= 2 also
 *     use the handle's split-K workspace (partial tiles and per-tile
 *     counters): such calls on one handle must not overlap on the GPU --
 *     order them on one stream; calls on different handles are independent.
 */
#ifndef SGEMV_H
#define SGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sgemv_ctx* sgemv_t;

enum {
  SGEMV_OK = 0,
  SGEMV_ERR_ARG = -1,         /* bad argument: shape, pointer, alignment, m */
  SGEMV_ERR_UNSUPPORTED = -2, /* valid request this build does not support */
  SGEMV_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  SGEMV_ERR_STATE = -4,       /* run/export before pack or import */
  SGEMV_ERR_TIMEOUT = -5,     /* a bounded device-side wait gave up */
  SGEMV_ERR_NONFINITE = -6,   /* NaN or Inf in the weight given to pack */
  SGEMV_ERR_RANGE = -7        /* a group's scale does not fit binary16 */
};

/* Size limits of one handle. */
#define SGEMV_MAX_ROWS (1 << 24)
#define SGEMV_MAX_COLS (1 << 20)
#define SGEMV_MAX_M 64

/*
 * Create a handle for a rows x cols weight with N = n_keep (1 or 2) kept per
 * quad and group size `group` (64, 128 or 256 dense columns; cols must be a
 * multiple of it).  rows and cols may be 0 (empty products).  max_m (1..64)
 * bounds the activation rows of later runs.  `device` is the CUDA ordinal.
 * Allocates the packed-weight buffers on that device; nothing is packed yet.
 * On failure *out is set to NULL.
 */
int sgemv_create(sgemv_t* out, int rows, int cols, int n_keep, int group,
                 int max_m, int device);

/*
 * As sgemv_create, with a group size per row instead of per matrix: the
 * paper gives sensitive channels more (finer) groups inside one layer
 * (section 3.2, "Adaptive group quantization").  row_group (host, rows
 * entries, read only) holds each row's group size, 64, 128 or 256, each a
 * divisor of cols.  Row r is quantised exactly as a one-row matrix with
 * group row_group[r].  The canonical scale and zero arrays of import and
 * export are then flat: row r's cols / row_group[r] entries follow those of
 * rows 0..r-1 (sgemv_sizes reports their total).  Every other call works as
 * for sgemv_create.  In device memory the scale/zero words are kept at the
 * finest group of the matrix, a coarser group's pair repeated in each of its
 * sub-groups, so a product reads 4 * cols / min(row_group) bytes of them per
 * row; sgemv_packed_bytes counts the canonical ones.
 */
int sgemv_create_rowgroups(sgemv_t* out, int rows, int cols, int n_keep,
                           const int* row_group, int max_m, int device);

/*
 * Prune, quantise and pack a dense fp32 weight (rows x cols, row-major,
 * host memory, read only).  The work runs on the handle's device; the call
 * returns when it is done.  NaN/Inf anywhere -> SGEMV_ERR_NONFINITE; a scale
 * beyond binary16 -> SGEMV_ERR_RANGE; the handle is then left unpacked.
 */
int sgemv_pack(sgemv_t h, const float* w_host);

/* As sgemv_pack, with the dense weight already in device memory; the work is
 * ordered on `stream`, and the call waits for it before returning. */
int sgemv_pack_device(sgemv_t h, const float* w_dev, void* stream);

/*
 * As sgemv_pack, but each quad keeps the N weights of largest importance
 * score, the pruning criterion of the paper (section 3.2, "Sparsification",
 * Eq. 3):
 *   score_ij = |W_ij| * xnorm[j] + |W_ij| * |grad_ij|,
 * evaluated in binary32 as written (two products and one sum, each rounded
 * to nearest once), ties to the lower column.  Quantisation is unchanged.
 *   xnorm_host : cols values, the L2 norm of input channel j over the
 *                caller's calibration activations; finite and >= 0
 *                (SGEMV_ERR_NONFINITE / SGEMV_ERR_ARG otherwise);
 *   grad_host  : rows x cols row-major, the loss gradient dE/dW, or NULL for
 *                a zero gradient; NaN/Inf -> SGEMV_ERR_NONFINITE.
 * All three host arrays are read only.  With every norm equal to a power of
 * two and no gradient the result equals sgemv_pack's.  Synchronous.
 */
int sgemv_pack_scored(sgemv_t h, const float* w_host, const float* xnorm_host,
                      const float* grad_host);

/*
 * Load canonical 2bit-CSR bytes (host memory, layout above; the byte counts
 * are those reported by sgemv_sizes).  For N = 2 the two positions of each
 * quad must ascend strictly (SGEMV_ERR_ARG otherwise).  Synchronous.
 */
int sgemv_import(sgemv_t h, const uint8_t* vals, const uint8_t* idx,
                 const uint16_t* scale, const uint16_t* zero);

/* Write the packed weight back as canonical bytes into host buffers of the
 * sizes reported by sgemv_sizes.  Synchronous. */
int sgemv_export(sgemv_t h, uint8_t* vals, uint8_t* idx, uint16_t* scale,
                 uint16_t* zero);

/*
 * y = W_hat . x for m activation rows (0 <= m <= max_m).  m = 1 runs the
 * CUDA-core decode kernel; batches (beam candidates, prefix-tree
 * verification nodes: the paper's parallel verification, section 3.1) run
 * on the sparse tensor cores with the 2-bit positions as the MMA's 2:4
 * metadata -- 2 <= m <= 32 with the warp-level sparse MMA, 33 <= m <= 64
 * with tcgen05 and the accumulators in tensor memory.
 *   x_dev : m x cols binary16, row-major, 16-byte aligned, device memory;
 *   y_dev : m x rows binary16, row-major, 2-byte aligned, device memory,
 *           fully overwritten; must not overlap x_dev;
 *   accumulation is fp32, each y element rounded once to binary16.
 * Asynchronous on `stream`: returns after the launch, reporting argument
 * and launch errors only.  The handle must have been packed or imported.
 * cols = 0 writes y = +0.  A matrix whose device layout holds 2^31 or more
 * 32-weight chunks or scale/zero words (48 GiB or more of packed weight)
 * -> SGEMV_ERR_UNSUPPORTED.
 */
int sgemv_run(sgemv_t h, const void* x_dev, void* y_dev, int m, void* stream);

/*
 * The same product with x and y in host memory: the call copies x to a
 * staging buffer owned by the handle, runs, and copies y back, all ordered
 * on `stream`; it returns without waiting, so the caller synchronises the
 * stream before reading y_host.  Page-locked host buffers make the copies
 * asynchronous.  Calls on one handle share its staging buffers and must be
 * ordered on one stream.
 */
int sgemv_run_host(sgemv_t h, const void* x_host, void* y_host, int m,
                   void* stream);

/*
 * Several products that share one activation x -- e.g. the q, k and v
 * projections of a decoder layer, or its gate and up projections -- as
 * y_i = W_hat_i . x for i < count.  This is the grouped run of the
 * layer's decode step (the paper's kernel serves every linear layer of the
 * decode, section 1 contribution 2): with m = 1 the matrices go into one
 * launch -- at most 8 of each N; the CTAs of one part take the 2:4 matrices
 * and those of the other the 1:4 ones, in proportion to their packed bytes,
 * and each CTA stages x and its lookup table once for all of its matrices
 * (more than 8 of one N: one launch per N and per 8).  With 2 <= m <= 32 the
 * matrices of one N share a launch of the batch kernel (at most 8 per
 * launch) when their row tiles still leave room to split K across a
 * cluster, else each runs alone; the outputs then match a single run within
 * the same tolerance, but the order of the fp32 partial sums may differ.
 * A device-side error of a shared launch (a bounded wait that ran out) is
 * recorded in the status word of the launch's first handle.  With
 * 33 <= m <= 64 the matrices of one N and group size share a launch of the
 * tensor-core batch kernel (at most 4 per launch; the split-K partials use
 * the first handle's workspace).
 *   handles : count packed handles on one device, all with the same cols;
 *             n_keep and group may differ;
 *   x_dev   : m x cols binary16, 16-byte aligned, shared by all;
 *   y_devs  : count device pointers, y_devs[i] is m x rows_i binary16,
 *             2-byte aligned, none overlapping x_dev or one another
 *             (SGEMV_ERR_ARG otherwise);
 *   m       : 0 <= m <= every handle's max_m.
 * Asynchronous on `stream`, like sgemv_run; count = 0 is a no-op.  The
 * next work on the stream sees every y_i complete.
 */
int sgemv_run_group(const sgemv_t* handles, int count, const void* x_dev,
                    void* const* y_devs, int m, void* stream);

/*
 * The grouped run with x and the outputs in host memory, as sgemv_run_host
 * is to sgemv_run: x_host (m x cols binary16) is copied to the first
 * handle's staging buffer, the products run as in sgemv_run_group into each
 * handle's own output staging, and y_i goes back to y_hosts[i] (m x rows_i
 * binary16), all ordered on `stream`; the call returns without waiting, so
 * the caller synchronises the stream before reading the outputs.  A handle
 * may appear only once (SGEMV_ERR_ARG otherwise); calls that share a handle
 * must be ordered on one stream.  Page-locked host buffers make the copies
 * asynchronous.
 */
int sgemv_run_group_host(const sgemv_t* handles, int count, const void* x_host,
                         void* const* y_hosts, int m, void* stream);

/*
 * sgemv_run for 2 <= m <= min(64, max_m) that allocates nothing (the paper
 * has no counterpart: this is a deployment variant).  Meant for callers
 * that may not allocate device memory when they run the product: code under
 * an allocator that owns all device memory (an arena reserved at start-up,
 * a framework that must account for every byte) and plug-ins handed their
 * buffers but no right to allocate.  The product, arguments and result are
 * those of sgemv_run; the difference is where the batch kernel's split-K
 * workspace lives: instead of the handle's own (allocated by sgemv_create
 * when max_m >= 2), a fixed array inside the library -- 10 MiB of fp32
 * partial tiles plus 64 KiB of per-tile counters -- that every GPU which
 * loads the library holds until the process exits.  It runs the tcgen05
 * batch kernel at every m (sgemv_run takes the warp-level one for m <= 32),
 * so for those m the order of the fp32 partial sums, not the tolerance, may
 * differ from sgemv_run's.  Limits: at most
 * 2,097,152 weight rows (16384 row tiles of 128) -> SGEMV_ERR_UNSUPPORTED
 * beyond; m outside [2, min(64, max_m)] -> SGEMV_ERR_ARG (m = 1 needs no
 * workspace: use sgemv_run).  The handle may have been created with any
 * max_m >= 2.  Every call shares the one array per device and each call
 * clears its counters first: calls that overlap on the GPU race, so order
 * them on one stream (they may overlap with sgemv_run calls, which use the
 * handles' own workspaces).  The first call on a device looks up the
 * array's device address once, with that device current.  Asynchronous on
 * `stream`, like sgemv_run.
 */
int sgemv_run_noalloc(sgemv_t h, const void* x_dev, void* y_dev, int m, void* stream);

/* Synchronise the device, then return and clear the handle's device error
 * word (SGEMV_OK if no kernel reported an error since the last call).  A
 * batch kernel reports SGEMV_ERR_TIMEOUT when one of its bounded waits gave
 * up after about a second; the outputs of that call are then undefined and
 * later calls are unaffected.  2 <= m <= 8: the split-K reduction waiting
 * for the partial sums of the other CTAs of its cluster -- every CTA still
 * issues all of its sends and no CTA retires before every CTA of its cluster
 * has issued them, so no late store lands in a retired CTA; what the limit
 * cannot guard against is a CTA that never reaches its sends (the launch
 * then does not finish).  9 <= m <= 32 reduce between cluster barriers that
 * every CTA reaches, with no such wait.  33 <= m <= 64: the waits for
 * its own TMA copies and MMAs -- it then stops issuing work, lets the copies
 * it issued land, frees its tensor memory and completes its split-K
 * counters. */
int sgemv_status(sgemv_t h);

/*
 * Failure-detection test hook (not a paper operation).  The next `runs`
 * batch products on this handle with 2 <= m <= 8 or 33 <= m <= 64 make
 * their bounded wait run out: for 2 <= m <= 8 every cluster rank withholds
 * its split-K partial sums, for m >= 33 the kernel withholds its x copies,
 * and the wait limit drops to about 20 microseconds.  sgemv_status then
 * returns SGEMV_ERR_TIMEOUT and y of those calls is undefined.  Nothing the
 * kernel waits for is in flight when it gives up, the device stays usable
 * and later calls run normally.  Calls with m = 1 or 9 <= m <= 32 (whose
 * kernels wait on no copy, only on cluster barriers) do not consume the
 * hook.
 * runs = 0 cancels; runs < 0 -> SGEMV_ERR_ARG.
 */
int sgemv_debug_withhold(sgemv_t h, int runs);

/*
 * Byte counts of the canonical arrays and of the device-resident packed
 * weight.  Any output pointer may be NULL.
 */
int sgemv_sizes(sgemv_t h, size_t* vals_bytes, size_t* idx_bytes,
                size_t* n_groups, size_t* device_bytes);

/* Algorithmic packed-weight bytes: INT4 values + 2-bit positions + binary16
 * scale and zero per group (0 for a NULL handle). */
size_t sgemv_packed_bytes(sgemv_t h);

/* Text of the calling thread's last error ("" if none). */
const char* sgemv_last_error(void);

/* Free the handle and its device buffers.  NULL is accepted. */
int sgemv_destroy(sgemv_t h);

#ifdef __cplusplus
}
#endif

#endif /* SGEMV_H */
