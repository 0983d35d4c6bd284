// sgemv_api.cu -- the extern "C" boundary of libsgemv (declared in
// include/sgemv.h): argument checks, handle and device-buffer management,
// host<->device transfers, and kernel dispatch.  No arithmetic of the
// method happens here; every step of pack and run executes in the CUDA
// kernels of sgemv_format.cu, sgemv_m1.cu and sgemv_mma.cu.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cmath>

#include "sgemv_internal.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SGEMV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CUDA_TRY(expr, what)                       \
  do {                                             \
    cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Makes the handle's device current for the scope and restores the caller's.
struct DeviceGuard {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

// A device buffer freed on scope exit (used for pack / import / export
// temporaries).
struct DevBuf {
  void* p = nullptr;
  ~DevBuf() {
    if (p) cudaFree(p);
  }
  cudaError_t alloc(size_t n) { return n ? cudaMalloc(&p, n) : cudaSuccess; }
};

sgemv::Layout make_layout(int rows, int cols, int n_keep, int group) {
  sgemv::Layout L;
  L.rows = rows;
  L.cols = cols;
  L.n_keep = n_keep;
  L.group = group;
  L.kept = (int64_t)cols / 4 * n_keep;
  L.chunks = (L.kept + sgemv::kChunkKept - 1) / sgemv::kChunkKept;
  L.cstride = (L.chunks + 1) & ~(int64_t)1;
  L.ngroups = cols / group;
  L.gstride = (L.ngroups + 3) & ~(int64_t)3;
  L.vals_row = (L.kept + 1) / 2;
  L.idx_row = (L.kept + 3) / 4;
  return L;
}

int check_handle(sgemv_t h) {
  if (!h) return fail(SGEMV_ERR_ARG, "null handle");
  return SGEMV_OK;
}

int dev_err_to_status(int word) {
  switch (word) {
    case 0: return SGEMV_OK;
    case sgemv::kDevErrNonfinite:
      return fail(SGEMV_ERR_NONFINITE, "weight holds NaN or Inf");
    case sgemv::kDevErrRange:
      return fail(SGEMV_ERR_RANGE, "a group's scale does not fit binary16");
    case sgemv::kDevErrBadIndex:
      return fail(SGEMV_ERR_ARG, "2:4 positions must ascend strictly within a quad");
    case sgemv::kDevErrTimeout:
      return fail(SGEMV_ERR_TIMEOUT,
                  "a bounded device wait gave up: a batch kernel's copies, MMAs or split-K "
                  "partial sums did not arrive in time; the outputs of that call are undefined");
    case sgemv::kDevErrChecked:
      return fail(SGEMV_ERR_ARG,
                  "checked build: a product kernel decoded a 2:4 position pair that does not "
                  "ascend, or an index outside its row (the packed weight is corrupt)");
    default:
      return fail(SGEMV_ERR_CUDA, "device error word %d", word);
  }
}

// Reads and clears the error word after the handle's private stream drains.
int collect_dev_err(sgemv_t h) {
  CUDA_TRY(cudaStreamSynchronize(h->stream), "cudaStreamSynchronize");
  int word = 0;
  CUDA_TRY(cudaMemcpy(&word, h->d_err, sizeof word, cudaMemcpyDeviceToHost),
           "read error word");
  CUDA_TRY(cudaMemset(h->d_err, 0, sizeof(int)), "clear error word");
  return dev_err_to_status(word);
}

size_t vals_dev_bytes(const sgemv::Layout& L) { return (size_t)L.rows * L.cstride * 16; }
size_t idx_dev_bytes(const sgemv::Layout& L) { return (size_t)L.rows * L.cstride * 8; }
size_t sz_dev_bytes(const sgemv::Layout& L) { return (size_t)L.rows * L.gstride * 4; }

sgemv::RowGroups row_groups(sgemv_t h) {
  sgemv::RowGroups g;
  g.rowg = h->d_rowg;
  g.goff = h->d_goff;
  return g;
}

void free_ctx(sgemv_t h) {
  if (!h) return;
  cudaFree(h->d_vals);
  cudaFree(h->d_idx);
  cudaFree(h->d_sz);
  cudaFree(h->d_xstage);
  cudaFree(h->d_ystage);
  cudaFree(h->d_err);
  cudaFree(h->d_rowg);
  cudaFree(h->d_goff);
  cudaFree(h->tc.scratch);
  cudaFree(h->tc.counters);
  if (h->stream) cudaStreamDestroy(h->stream);
  delete h;
}

int pack_on_device(sgemv_t h, const float* w_dev, cudaStream_t s, const float* xnorm_dev = nullptr,
                   const float* grad_dev = nullptr) {
  const sgemv::Layout& L = h->L;
  h->ready = false;
  CUDA_TRY(cudaMemsetAsync(h->d_err, 0, sizeof(int), s), "clear error word");
  if (vals_dev_bytes(L))
    CUDA_TRY(cudaMemsetAsync(h->d_vals, 0, vals_dev_bytes(L), s), "memset vals");
  if (idx_dev_bytes(L))
    CUDA_TRY(cudaMemsetAsync(h->d_idx, 0, idx_dev_bytes(L), s), "memset idx");
  if (sz_dev_bytes(L))
    CUDA_TRY(cudaMemsetAsync(h->d_sz, 0, sz_dev_bytes(L), s), "memset scale/zero");
  CUDA_TRY(sgemv::launch_pack(L, row_groups(h), w_dev, xnorm_dev, grad_dev, h->d_vals, h->d_idx, h->d_sz,
                              h->d_err, s),
           "pack kernel");
  CUDA_TRY(cudaStreamSynchronize(s), "pack");
  int word = 0;
  CUDA_TRY(cudaMemcpy(&word, h->d_err, sizeof word, cudaMemcpyDeviceToHost),
           "read error word");
  CUDA_TRY(cudaMemset(h->d_err, 0, sizeof(int)), "clear error word");
  int rc = dev_err_to_status(word);
  if (rc == SGEMV_OK) h->ready = true;
  return rc;
}

}  // namespace

extern "C" {

const char* sgemv_last_error(void) { return g_err; }

}  // extern "C"

namespace sgemv {
// Status reporting for the library's other translation units: the same
// thread-local text that sgemv_last_error returns.
int report(int code, const char* msg) { return fail(code, "%s", msg); }
int report_cuda(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace sgemv

// Creates a handle; row_group (host, rows entries) optional.
static int create_impl(sgemv_t* out, int rows, int cols, int n_keep, int group,
                       const int* row_group, int max_m, int device) {
  if (!out) return fail(SGEMV_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (rows < 0 || rows > SGEMV_MAX_ROWS)
    return fail(SGEMV_ERR_ARG, "rows=%d outside [0, %d]", rows, SGEMV_MAX_ROWS);
  if (cols < 0 || cols > SGEMV_MAX_COLS)
    return fail(SGEMV_ERR_ARG, "cols=%d outside [0, %d]", cols, SGEMV_MAX_COLS);
  if (n_keep != 1 && n_keep != 2)
    return fail(SGEMV_ERR_ARG, "n_keep=%d: only 1:4 and 2:4 are defined", n_keep);
  if (group != 64 && group != 128 && group != 256)
    return fail(SGEMV_ERR_ARG, "group=%d: must be 64, 128 or 256", group);
  if (cols % group != 0)
    return fail(SGEMV_ERR_ARG, "cols=%d is not a multiple of group=%d", cols, group);
  if (max_m < 1 || max_m > SGEMV_MAX_M)
    return fail(SGEMV_ERR_ARG, "max_m=%d outside [1, %d]", max_m, SGEMV_MAX_M);
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device < 0 || device >= ndev)
    return fail(SGEMV_ERR_ARG, "device=%d but %d device(s) visible", device, ndev);
  DeviceGuard g(device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");

  sgemv_t h = new sgemv_ctx();
  memset(h, 0, sizeof *h);
  h->L = make_layout(rows, cols, n_keep, group);
  h->canon_groups = (int64_t)rows * h->L.ngroups;
  h->max_m = max_m;
  h->device = device;
  h->ready = false;
  auto try_alloc = [&](void** p, size_t n, const char* what) -> int {
    if (n == 0) return SGEMV_OK;
    cudaError_t err = cudaMalloc(p, n);
    if (err != cudaSuccess) return cuda_fail(err, what);
    return SGEMV_OK;
  };
  int rc = SGEMV_OK;
  if (!rc) rc = try_alloc((void**)&h->d_vals, vals_dev_bytes(h->L), "cudaMalloc vals");
  if (!rc) rc = try_alloc((void**)&h->d_idx, idx_dev_bytes(h->L), "cudaMalloc idx");
  if (!rc) rc = try_alloc((void**)&h->d_sz, sz_dev_bytes(h->L), "cudaMalloc scale/zero");
  if (!rc) rc = try_alloc((void**)&h->d_xstage, (size_t)max_m * cols * 2, "cudaMalloc x staging");
  if (!rc) rc = try_alloc((void**)&h->d_ystage, (size_t)max_m * rows * 2, "cudaMalloc y staging");
  if (!rc) rc = try_alloc((void**)&h->d_err, sizeof(int), "cudaMalloc error word");
  if (!rc) {
    e = cudaMemset(h->d_err, 0, sizeof(int));
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemset");
  }
  if (!rc) {
    e = cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaStreamCreate");
  }
  if (!rc && row_group && rows > 0) {
    // group size per row: device copy and the canonical scale/zero offsets
    int64_t* off = new int64_t[(size_t)rows + 1];
    off[0] = 0;
    for (int r = 0; r < rows; ++r) off[r + 1] = off[r] + cols / row_group[r];
    h->canon_groups = off[rows];
    rc = try_alloc((void**)&h->d_rowg, (size_t)rows * sizeof(int), "cudaMalloc row groups");
    if (!rc) rc = try_alloc((void**)&h->d_goff, ((size_t)rows + 1) * sizeof(int64_t),
                            "cudaMalloc group offsets");
    if (!rc) {
      e = cudaMemcpy(h->d_rowg, row_group, (size_t)rows * sizeof(int), cudaMemcpyHostToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy(h->d_goff, off, ((size_t)rows + 1) * sizeof(int64_t),
                       cudaMemcpyHostToDevice);
      if (e != cudaSuccess) rc = cuda_fail(e, "copy row groups");
    }
    delete[] off;
  }
  if (!rc && max_m >= 2 && rows > 0 && cols > 0) {
    // the tensor-core batch kernel: split-K workspace, zeroed per-tile
    // arrival counters, and tensor maps of the packed weight
    rc = try_alloc((void**)&h->tc.scratch, sgemv::tc_scratch_bytes(max_m),
                   "cudaMalloc split-K workspace");
    const size_t cnt = (size_t)sgemv::tc_tiles(h->L) * sizeof(int);
    if (!rc) rc = try_alloc((void**)&h->tc.counters, cnt, "cudaMalloc split-K counters");
    if (!rc) {
      e = cudaMemset(h->tc.counters, 0, cnt);
      if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemset");
    }
    if (!rc) {
      h->tc.ready = sgemv::tc_encode_weights(h->L, h->d_vals, h->d_idx, h->d_sz, &h->tc);
      if (!h->tc.ready)
        rc = fail(SGEMV_ERR_CUDA, "encoding the tensor maps of the packed weight failed");
    }
  }
  if (rc) {
    free_ctx(h);
    return rc;
  }
  *out = h;
  return SGEMV_OK;
}

extern "C" {

int sgemv_create(sgemv_t* out, int rows, int cols, int n_keep, int group,
                 int max_m, int device) {
  return create_impl(out, rows, cols, n_keep, group, nullptr, max_m, device);
}

int sgemv_create_rowgroups(sgemv_t* out, int rows, int cols, int n_keep,
                           const int* row_group, int max_m, int device) {
  if (!out) return fail(SGEMV_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (rows < 0 || rows > SGEMV_MAX_ROWS)
    return fail(SGEMV_ERR_ARG, "rows=%d outside [0, %d]", rows, SGEMV_MAX_ROWS);
  if (rows > 0 && !row_group) return fail(SGEMV_ERR_ARG, "row_group is NULL");
  int gmin = rows > 0 ? 256 : 64;
  for (int r = 0; r < rows; ++r) {
    const int g = row_group[r];
    if (g != 64 && g != 128 && g != 256)
      return fail(SGEMV_ERR_ARG, "row_group[%d]=%d: must be 64, 128 or 256", r, g);
    if (cols % g != 0)
      return fail(SGEMV_ERR_ARG, "cols=%d is not a multiple of row_group[%d]=%d", cols, r, g);
    gmin = g < gmin ? g : gmin;
  }
  return create_impl(out, rows, cols, n_keep, gmin, row_group, max_m, device);
}

int sgemv_destroy(sgemv_t h) {
  if (!h) return SGEMV_OK;
  DeviceGuard g(h->device);
  free_ctx(h);
  return SGEMV_OK;
}

int sgemv_pack(sgemv_t h, const float* w_host) {
  if (int rc = check_handle(h)) return rc;
  const sgemv::Layout& L = h->L;
  const size_t n = (size_t)L.rows * L.cols;
  if (n && !w_host) return fail(SGEMV_ERR_ARG, "w_host is NULL");
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  DevBuf w;
  CUDA_TRY(w.alloc(n * sizeof(float)), "cudaMalloc dense weight");
  if (n)
    CUDA_TRY(cudaMemcpyAsync(w.p, w_host, n * sizeof(float), cudaMemcpyHostToDevice,
                             h->stream),
             "copy weight to device");
  return pack_on_device(h, static_cast<const float*>(w.p), h->stream);
}

int sgemv_pack_scored(sgemv_t h, const float* w_host, const float* xnorm_host,
                      const float* grad_host) {
  if (int rc = check_handle(h)) return rc;
  const sgemv::Layout& L = h->L;
  const size_t n = (size_t)L.rows * L.cols;
  if (n && !w_host) return fail(SGEMV_ERR_ARG, "w_host is NULL");
  if (L.cols && !xnorm_host) return fail(SGEMV_ERR_ARG, "xnorm_host is NULL");
  for (int c = 0; c < L.cols; ++c) {
    if (!std::isfinite(xnorm_host[c]))
      return fail(SGEMV_ERR_NONFINITE, "xnorm[%d] is not finite", c);
    if (xnorm_host[c] < 0.0f) return fail(SGEMV_ERR_ARG, "xnorm[%d] is negative", c);
  }
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  DevBuf w, xn, gr;
  CUDA_TRY(w.alloc(n * sizeof(float)), "cudaMalloc dense weight");
  CUDA_TRY(xn.alloc((size_t)L.cols * sizeof(float)), "cudaMalloc norms");
  if (grad_host) CUDA_TRY(gr.alloc(n * sizeof(float)), "cudaMalloc gradient");
  if (n) {
    CUDA_TRY(cudaMemcpyAsync(w.p, w_host, n * sizeof(float), cudaMemcpyHostToDevice, h->stream),
             "copy weight to device");
    if (grad_host)
      CUDA_TRY(cudaMemcpyAsync(gr.p, grad_host, n * sizeof(float), cudaMemcpyHostToDevice,
                               h->stream),
               "copy gradient to device");
  }
  if (L.cols)
    CUDA_TRY(cudaMemcpyAsync(xn.p, xnorm_host, (size_t)L.cols * sizeof(float),
                             cudaMemcpyHostToDevice, h->stream),
             "copy norms to device");
  return pack_on_device(h, static_cast<const float*>(w.p), h->stream,
                        static_cast<const float*>(xn.p), static_cast<const float*>(gr.p));
}

int sgemv_pack_device(sgemv_t h, const float* w_dev, void* stream) {
  if (int rc = check_handle(h)) return rc;
  const size_t n = (size_t)h->L.rows * h->L.cols;
  if (n && !w_dev) return fail(SGEMV_ERR_ARG, "w_dev is NULL");
  if (n && ((uintptr_t)w_dev & 15u))
    return fail(SGEMV_ERR_ARG, "w_dev must be 16-byte aligned");
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  return pack_on_device(h, w_dev, static_cast<cudaStream_t>(stream));
}

int sgemv_import(sgemv_t h, const uint8_t* vals, const uint8_t* idx,
                 const uint16_t* scale, const uint16_t* zero) {
  if (int rc = check_handle(h)) return rc;
  const sgemv::Layout& L = h->L;
  const size_t nv = (size_t)L.rows * L.vals_row, ni = (size_t)L.rows * L.idx_row;
  const size_t ns = (size_t)h->canon_groups;
  if ((nv && !vals) || (ni && !idx) || (ns && (!scale || !zero)))
    return fail(SGEMV_ERR_ARG, "a canonical input pointer is NULL");
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  h->ready = false;
  DevBuf cv, ci, cs, cz;
  CUDA_TRY(cv.alloc(nv), "cudaMalloc");
  CUDA_TRY(ci.alloc(ni), "cudaMalloc");
  CUDA_TRY(cs.alloc(ns * 2), "cudaMalloc");
  CUDA_TRY(cz.alloc(ns * 2), "cudaMalloc");
  cudaStream_t s = h->stream;
  if (nv) CUDA_TRY(cudaMemcpyAsync(cv.p, vals, nv, cudaMemcpyHostToDevice, s), "copy vals");
  if (ni) CUDA_TRY(cudaMemcpyAsync(ci.p, idx, ni, cudaMemcpyHostToDevice, s), "copy idx");
  if (ns) {
    CUDA_TRY(cudaMemcpyAsync(cs.p, scale, ns * 2, cudaMemcpyHostToDevice, s), "copy scale");
    CUDA_TRY(cudaMemcpyAsync(cz.p, zero, ns * 2, cudaMemcpyHostToDevice, s), "copy zero");
  }
  CUDA_TRY(cudaMemsetAsync(h->d_err, 0, sizeof(int), s), "clear error word");
  if (sz_dev_bytes(L))
    CUDA_TRY(cudaMemsetAsync(h->d_sz, 0, sz_dev_bytes(L), s), "memset scale/zero");
  CUDA_TRY(sgemv::launch_canon_to_device(
               L, row_groups(h), (const uint8_t*)cv.p, (const uint8_t*)ci.p, (const uint16_t*)cs.p,
               (const uint16_t*)cz.p, h->d_vals, h->d_idx, h->d_sz, h->d_err, s),
           "import kernel");
  int rc = collect_dev_err(h);
  if (rc == SGEMV_OK) h->ready = true;
  return rc;
}

int sgemv_export(sgemv_t h, uint8_t* vals, uint8_t* idx, uint16_t* scale,
                 uint16_t* zero) {
  if (int rc = check_handle(h)) return rc;
  if (!h->ready) return fail(SGEMV_ERR_STATE, "export before pack or import");
  const sgemv::Layout& L = h->L;
  const size_t nv = (size_t)L.rows * L.vals_row, ni = (size_t)L.rows * L.idx_row;
  const size_t ns = (size_t)h->canon_groups;
  if ((nv && !vals) || (ni && !idx) || (ns && (!scale || !zero)))
    return fail(SGEMV_ERR_ARG, "a canonical output pointer is NULL");
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  DevBuf cv, ci, cs, cz;
  CUDA_TRY(cv.alloc(nv), "cudaMalloc");
  CUDA_TRY(ci.alloc(ni), "cudaMalloc");
  CUDA_TRY(cs.alloc(ns * 2), "cudaMalloc");
  CUDA_TRY(cz.alloc(ns * 2), "cudaMalloc");
  cudaStream_t s = h->stream;
  CUDA_TRY(sgemv::launch_device_to_canon(L, row_groups(h), h->d_vals, h->d_idx, h->d_sz,
                                         (uint8_t*)cv.p, (uint8_t*)ci.p,
                                         (uint16_t*)cs.p, (uint16_t*)cz.p, s),
           "export kernel");
  if (nv) CUDA_TRY(cudaMemcpyAsync(vals, cv.p, nv, cudaMemcpyDeviceToHost, s), "copy vals");
  if (ni) CUDA_TRY(cudaMemcpyAsync(idx, ci.p, ni, cudaMemcpyDeviceToHost, s), "copy idx");
  if (ns) {
    CUDA_TRY(cudaMemcpyAsync(scale, cs.p, ns * 2, cudaMemcpyDeviceToHost, s), "copy scale");
    CUDA_TRY(cudaMemcpyAsync(zero, cz.p, ns * 2, cudaMemcpyDeviceToHost, s), "copy zero");
  }
  CUDA_TRY(cudaStreamSynchronize(s), "export");
  return SGEMV_OK;
}

static int run_checked(sgemv_t h, const void* x, void* y, int m, cudaStream_t s) {
  const sgemv::Layout& L = h->L;
  sgemv::RunArgs a;
  a.vals = h->d_vals;
  a.idx = h->d_idx;
  a.sz = h->d_sz;
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.m = m;
  a.err = h->d_err;
  if (m == 0 || L.rows == 0) return SGEMV_OK;
  if (h->withhold_runs > 0 && sgemv::withhold_applies(L, m)) {
    a.withhold = 1;
    --h->withhold_runs;
  }
  // cols = 0: every output is the empty sum, +0
  if (L.cols == 0) {
    CUDA_TRY(cudaMemsetAsync(a.y, 0, (size_t)m * L.rows * sizeof(__half), s), "zero y");
    return SGEMV_OK;
  }
  // m = 1: the CUDA-core pair-table kernel; 2 <= m <= mma_max_m(N) (32): the
  // warp-level sparse MMA kernel; up to 64: the tcgen05 kernel (each
  // measured the fastest in its range on the 7B layer shapes)
  cudaError_t e = m == 1                       ? sgemv::launch_m1(L, a, s)
                  : m <= sgemv::mma_max_m(L.n_keep) ? sgemv::launch_mma(L, a, s)
                                             : sgemv::launch_tc(L, a, h->tc, s);
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    return fail(SGEMV_ERR_UNSUPPORTED,
                "a %d x %d matrix is beyond the product kernels' 32-bit chunk index space",
                L.rows, L.cols);
  }
  if (e != cudaSuccess) return cuda_fail(e, "SparseGemv launch");
  return SGEMV_OK;
}

static int run_args_ok(sgemv_t h, const void* x, const void* y, int m) {
  if (int rc = check_handle(h)) return rc;
  if (!h->ready) return fail(SGEMV_ERR_STATE, "run before pack or import");
  if (m < 0 || m > h->max_m)
    return fail(SGEMV_ERR_ARG, "m=%d outside [0, max_m=%d]", m, h->max_m);
  if (m > 0 && h->L.rows > 0) {
    if (!y) return fail(SGEMV_ERR_ARG, "y is NULL");
    if (h->L.cols > 0 && !x) return fail(SGEMV_ERR_ARG, "x is NULL");
  }
  return SGEMV_OK;
}

int sgemv_run(sgemv_t h, const void* x_dev, void* y_dev, int m, void* stream) {
  if (int rc = run_args_ok(h, x_dev, y_dev, m)) return rc;
  if (x_dev && ((uintptr_t)x_dev & 15u))
    return fail(SGEMV_ERR_ARG, "x_dev must be 16-byte aligned");
  if (y_dev && ((uintptr_t)y_dev & 1u))
    return fail(SGEMV_ERR_ARG, "y_dev must be 2-byte aligned");
  if (m > 0 && x_dev && y_dev) {
    const char* xb = static_cast<const char*>(x_dev);
    const char* yb = static_cast<const char*>(y_dev);
    const size_t xn = (size_t)m * h->L.cols * 2, yn = (size_t)m * h->L.rows * 2;
    if (xn && yn && xb < yb + yn && yb < xb + xn)
      return fail(SGEMV_ERR_ARG, "x and y overlap");
  }
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  return run_checked(h, x_dev, y_dev, m, static_cast<cudaStream_t>(stream));
}

int sgemv_run_host(sgemv_t h, const void* x_host, void* y_host, int m,
                   void* stream) {
  if (int rc = run_args_ok(h, x_host, y_host, m)) return rc;
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const sgemv::Layout& L = h->L;
  if (m == 0 || L.rows == 0) return SGEMV_OK;
  const size_t xn = (size_t)m * L.cols * 2, yn = (size_t)m * L.rows * 2;
  if (xn)
    CUDA_TRY(cudaMemcpyAsync(h->d_xstage, x_host, xn, cudaMemcpyHostToDevice, s),
             "copy x to device");
  if (int rc = run_checked(h, h->d_xstage, h->d_ystage, m, s)) return rc;
  CUDA_TRY(cudaMemcpyAsync(y_host, h->d_ystage, yn, cudaMemcpyDeviceToHost, s),
           "copy y to host");
  return SGEMV_OK;
}

static int run_group_checked(const sgemv_t* handles, int count, const void* x_dev,
                             void* const* y_devs, int m, cudaStream_t s);

int sgemv_run_group(const sgemv_t* handles, int count, const void* x_dev,
                    void* const* y_devs, int m, void* stream) {
  if (count < 0) return fail(SGEMV_ERR_ARG, "count=%d is negative", count);
  if (count == 0) return SGEMV_OK;
  if (!handles || !y_devs) return fail(SGEMV_ERR_ARG, "handles or y_devs is NULL");
  for (int i = 0; i < count; ++i) {
    if (int rc = run_args_ok(handles[i], x_dev, y_devs[i], m)) return rc;
    if (handles[i]->L.cols != handles[0]->L.cols)
      return fail(SGEMV_ERR_ARG, "handle %d has cols=%d, handle 0 has cols=%d", i,
                  handles[i]->L.cols, handles[0]->L.cols);
    if (handles[i]->device != handles[0]->device)
      return fail(SGEMV_ERR_ARG, "handles are on different devices");
    if (y_devs[i] && ((uintptr_t)y_devs[i] & 1u))
      return fail(SGEMV_ERR_ARG, "y_devs[%d] must be 2-byte aligned", i);
    if (m > 0 && x_dev && y_devs[i]) {
      const char* xb = static_cast<const char*>(x_dev);
      const char* yb = static_cast<const char*>(y_devs[i]);
      const size_t xn = (size_t)m * handles[i]->L.cols * 2;
      const size_t yn = (size_t)m * handles[i]->L.rows * 2;
      if (xn && yn && xb < yb + yn && yb < xb + xn)
        return fail(SGEMV_ERR_ARG, "x and y_devs[%d] overlap", i);
    }
  }
  // outputs must be disjoint (each is written by a different launch part)
  if (m > 0)
    for (int i = 0; i < count; ++i)
      for (int j = i + 1; j < count; ++j) {
        const char* a = static_cast<const char*>(y_devs[i]);
        const char* b = static_cast<const char*>(y_devs[j]);
        const size_t an = (size_t)m * handles[i]->L.rows * 2;
        const size_t bn = (size_t)m * handles[j]->L.rows * 2;
        if (a && b && an && bn && a < b + bn && b < a + an)
          return fail(SGEMV_ERR_ARG, "y_devs[%d] and y_devs[%d] overlap", i, j);
      }
  if (x_dev && ((uintptr_t)x_dev & 15u))
    return fail(SGEMV_ERR_ARG, "x_dev must be 16-byte aligned");
  DeviceGuard g(handles[0]->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  return run_group_checked(handles, count, x_dev, y_devs, m, static_cast<cudaStream_t>(stream));
}

// The grouped run after its arguments were checked, on the handles' device.
static int run_group_checked(const sgemv_t* handles, int count, const void* x_dev,
                             void* const* y_devs, int m, cudaStream_t s) {
  if (m == 0 || handles[0]->L.cols == 0) {
    for (int i = 0; i < count; ++i)
      if (int rc = run_checked(handles[i], x_dev, y_devs[i], m, s)) return rc;
    return SGEMV_OK;
  }
  if (m != 1) {
    bool hook = false;
    for (int i = 0; i < count; ++i) hook = hook || handles[i]->withhold_runs > 0;
    if (hook) {
      for (int i = 0; i < count; ++i)
        if (int rc = run_checked(handles[i], x_dev, y_devs[i], m, s)) return rc;
      return SGEMV_OK;
    }
    for (int n = 1; n <= 2; ++n) {
      if (m > sgemv::mma_max_m(n)) {
        // the tcgen05 kernel: one launch per group size and per
        // tc_max_group() matrices of this N
        const int tcap = sgemv::tc_max_group();
        for (int gs = 64; gs <= 256; gs *= 2) {
          sgemv::Layout Ls[8];
          sgemv::RunArgs as[8];
          const sgemv::TcMaps* maps[8];
          int k = 0;
          for (int i = 0; i <= count; ++i) {
            if (i < count && handles[i]->L.n_keep == n && handles[i]->L.group == gs &&
                handles[i]->L.rows > 0) {
              sgemv_t h = handles[i];
              Ls[k] = h->L;
              as[k].vals = h->d_vals;
              as[k].idx = h->d_idx;
              as[k].sz = h->d_sz;
              as[k].x = static_cast<const __half*>(x_dev);
              as[k].y = static_cast<__half*>(y_devs[i]);
              as[k].m = m;
              as[k].err = h->d_err;
              maps[k] = &h->tc;
              ++k;
            }
            if (k > 0 && (k == tcap || i == count)) {
              cudaError_t e = sgemv::launch_tc_group(Ls, as, maps, k, s, 1 << 30);
              if (e == cudaErrorNotSupported) {
                (void)cudaGetLastError();
                return fail(SGEMV_ERR_UNSUPPORTED,
                            "a grouped matrix is beyond the product kernels' 32-bit chunk index space");
              }
              if (e != cudaSuccess) return cuda_fail(e, "grouped SparseGemv launch");
              k = 0;
            }
          }
        }
        continue;
      }
      // the sparse MMA kernel: one launch per max_group() matrices of this N
      const int cap = sgemv::max_group();
      sgemv::Layout Ls[8];
      sgemv::RunArgs as[8];
      int k = 0;
      for (int i = 0; i <= count; ++i) {
        if (i < count && handles[i]->L.n_keep == n && handles[i]->L.rows > 0) {
          sgemv_t h = handles[i];
          Ls[k] = h->L;
          as[k].vals = h->d_vals;
          as[k].idx = h->d_idx;
          as[k].sz = h->d_sz;
          as[k].x = static_cast<const __half*>(x_dev);
          as[k].y = static_cast<__half*>(y_devs[i]);
          as[k].m = m;
          as[k].err = h->d_err;
          ++k;
        }
        if (k > 0 && (k == cap || i == count)) {
          cudaError_t e = sgemv::launch_mma_group(Ls, as, k, s);
          if (e == cudaErrorNotSupported) {
            (void)cudaGetLastError();
            return fail(SGEMV_ERR_UNSUPPORTED,
                        "a grouped matrix is beyond the product kernels' 32-bit chunk index space");
          }
          if (e != cudaSuccess) return cuda_fail(e, "grouped SparseGemv launch");
          k = 0;
        }
      }
    }
    return SGEMV_OK;
  }
  // m = 1: both N in one launch (two CTA ranges) when each fits a launch
  const int cap = sgemv::max_group();
  {
    sgemv::Layout L2[8], L1[8];
    sgemv::RunArgs a2[8], a1[8];
    int n2 = 0, n1 = 0;
    bool fits = true;
    for (int i = 0; i < count && fits; ++i) {
      sgemv_t h = handles[i];
      if (h->L.rows == 0) continue;
      const bool two = h->L.n_keep == 2;
      int& k = two ? n2 : n1;
      if (k == cap) {
        fits = false;
        break;
      }
      (two ? L2 : L1)[k] = h->L;
      sgemv::RunArgs& a = (two ? a2 : a1)[k];
      a.vals = h->d_vals;
      a.idx = h->d_idx;
      a.sz = h->d_sz;
      a.x = static_cast<const __half*>(x_dev);
      a.y = static_cast<__half*>(y_devs[i]);
      a.m = 1;
      a.err = h->d_err;
      ++k;
    }
    if (fits && n2 > 0 && n1 > 0) {
      cudaError_t e = sgemv::launch_m1_group_dual(L2, a2, n2, L1, a1, n1, s);
      if (e == cudaErrorNotSupported) {
        (void)cudaGetLastError();
        return fail(SGEMV_ERR_UNSUPPORTED,
                    "a grouped matrix is beyond the product kernels' 32-bit chunk index space");
      }
      if (e != cudaSuccess) return cuda_fail(e, "grouped SparseGemv launch");
      return SGEMV_OK;
    }
  }
  // otherwise one launch per N for up to max_group() matrices
  for (int n = 1; n <= 2; ++n) {
    sgemv::Layout Ls[8];
    sgemv::RunArgs as[8];
    int k = 0;
    for (int i = 0; i <= count; ++i) {
      const bool take = i < count && handles[i]->L.n_keep == n && handles[i]->L.rows > 0;
      if (take) {
        sgemv_t h = handles[i];
        Ls[k] = h->L;
        as[k].vals = h->d_vals;
        as[k].idx = h->d_idx;
        as[k].sz = h->d_sz;
        as[k].x = static_cast<const __half*>(x_dev);
        as[k].y = static_cast<__half*>(y_devs[i]);
        as[k].m = 1;
        as[k].err = h->d_err;
        ++k;
      }
      if (k > 0 && (k == cap || i == count)) {
        cudaError_t e = sgemv::launch_m1_group(Ls, as, k, s);
        if (e == cudaErrorNotSupported) {
          (void)cudaGetLastError();
          return fail(SGEMV_ERR_UNSUPPORTED,
                      "a grouped matrix is beyond the product kernels' 32-bit chunk index space");
        }
        if (e != cudaSuccess) return cuda_fail(e, "grouped SparseGemv launch");
        k = 0;
      }
    }
  }
  return SGEMV_OK;
}

int sgemv_run_group_host(const sgemv_t* handles, int count, const void* x_host,
                         void* const* y_hosts, int m, void* stream) {
  if (count < 0) return fail(SGEMV_ERR_ARG, "count=%d is negative", count);
  if (count == 0) return SGEMV_OK;
  if (!handles || !y_hosts) return fail(SGEMV_ERR_ARG, "handles or y_hosts is NULL");
  for (int i = 0; i < count; ++i) {
    if (int rc = run_args_ok(handles[i], x_host, y_hosts[i], m)) return rc;
    if (handles[i]->L.cols != handles[0]->L.cols)
      return fail(SGEMV_ERR_ARG, "handle %d has cols=%d, handle 0 has cols=%d", i,
                  handles[i]->L.cols, handles[0]->L.cols);
    if (handles[i]->device != handles[0]->device)
      return fail(SGEMV_ERR_ARG, "handles are on different devices");
    for (int j = 0; j < i; ++j)
      if (handles[j] == handles[i])
        return fail(SGEMV_ERR_ARG, "handle %d appears twice (its output staging is shared)", i);
  }
  DeviceGuard g(handles[0]->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (m == 0) return SGEMV_OK;
  // x into the first handle's staging buffer, the products into each
  // handle's own, y back to the caller
  const size_t xn = (size_t)m * handles[0]->L.cols * 2;
  if (xn)
    CUDA_TRY(cudaMemcpyAsync(handles[0]->d_xstage, x_host, xn, cudaMemcpyHostToDevice, s),
             "copy x to device");
  void* ys[64];
  void** yd = count <= 64 ? ys : new void*[count];
  for (int i = 0; i < count; ++i) yd[i] = handles[i]->d_ystage;
  int rc = run_group_checked(handles, count, handles[0]->d_xstage, yd, m, s);
  if (yd != ys) delete[] yd;
  if (rc) return rc;
  for (int i = 0; i < count; ++i) {
    const size_t yn = (size_t)m * handles[i]->L.rows * 2;
    if (yn)
      CUDA_TRY(cudaMemcpyAsync(y_hosts[i], handles[i]->d_ystage, yn, cudaMemcpyDeviceToHost, s),
               "copy y to host");
  }
  return SGEMV_OK;
}

int sgemv_debug_withhold(sgemv_t h, int runs) {
  if (int rc = check_handle(h)) return rc;
  if (runs < 0) return fail(SGEMV_ERR_ARG, "runs=%d is negative", runs);
  h->withhold_runs = runs;
  return SGEMV_OK;
}

int sgemv_status(sgemv_t h) {
  if (int rc = check_handle(h)) return rc;
  DeviceGuard g(h->device);
  if (g.err != cudaSuccess) return cuda_fail(g.err, "cudaSetDevice");
  CUDA_TRY(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  int word = 0;
  CUDA_TRY(cudaMemcpy(&word, h->d_err, sizeof word, cudaMemcpyDeviceToHost),
           "read error word");
  CUDA_TRY(cudaMemset(h->d_err, 0, sizeof(int)), "clear error word");
  return dev_err_to_status(word);
}

int sgemv_sizes(sgemv_t h, size_t* vals_bytes, size_t* idx_bytes,
                size_t* n_groups, size_t* device_bytes) {
  if (int rc = check_handle(h)) return rc;
  const sgemv::Layout& L = h->L;
  if (vals_bytes) *vals_bytes = (size_t)L.rows * L.vals_row;
  if (idx_bytes) *idx_bytes = (size_t)L.rows * L.idx_row;
  if (n_groups) *n_groups = (size_t)h->canon_groups;
  if (device_bytes) *device_bytes = vals_dev_bytes(L) + idx_dev_bytes(L) + sz_dev_bytes(L);
  return SGEMV_OK;
}

size_t sgemv_packed_bytes(sgemv_t h) {
  if (!h) return 0;
  const sgemv::Layout& L = h->L;
  const size_t kept = (size_t)L.rows * L.kept;
  return kept / 2 + kept / 4 + (size_t)h->canon_groups * 4;
}

}  // extern "C"
