// sgemv_noalloc.cu -- sgemv_run_noalloc: the batch product (2 <= m <= 64)
// for callers that cannot allocate device memory when they run it.
//
// Who cannot allocate: code that runs under an allocator owning all device
// memory (an arena reserved at start-up, or a framework whose caching
// allocator must account for every byte), and plug-ins that are handed their
// input and output buffers but no right to allocate.  The batch kernel needs
// a split-K workspace -- fp32 partial tiles of the row tiles that several
// CTAs share, and one arrival counter per row tile.  sgemv_run uses the
// handle's workspace, which sgemv_create allocates when max_m >= 2.  This
// entry point runs the same kernel on a workspace that is part of the
// library image instead: a file-scope __device__ array of fixed size, which
// every GPU that loads the library holds until the process exits.  The call
// itself allocates nothing (no cudaMalloc, no cudaFree, no allocating
// library routine).
#include <mutex>

#include "sgemv_internal.cuh"

namespace {

// The static workspace: 10 MiB of fp32 partial tiles (160 CTAs x 2 partial
// tiles x 128 rows x 64 columns) followed by 64 KiB of per-tile counters
// (16384 row tiles, i.e. up to 2,097,152 weight rows).
constexpr size_t kPartialBytes = (size_t)160 * 2 * 128 * 64 * sizeof(float);
constexpr size_t kCounterBytes = (size_t)16384 * sizeof(int);
constexpr int kMaxCtas = 160;
constexpr int kMaxTiles = 16384;

__device__ __align__(256) unsigned char g_noalloc_ws[kPartialBytes + kCounterBytes];

// Device address of g_noalloc_ws, looked up once per device.  In host code
// the array's name is only a host-side stand-in for the symbol: the kernel
// must be given the address that cudaGetSymbolAddress returns on the device
// that runs it.
std::mutex g_ws_lock;
void* g_ws_addr[64] = {nullptr};

cudaError_t workspace_address(int dev, void** out) {
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_ws_lock);
  if (!g_ws_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess) return e;
    g_ws_addr[dev] = p;
  }
  *out = g_ws_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

int sgemv_run_noalloc(sgemv_t h, const void* x_dev, void* y_dev, int m, void* stream) {
  if (!h) return sgemv::report(SGEMV_ERR_ARG, "null handle");
  if (!h->ready) return sgemv::report(SGEMV_ERR_STATE, "run before pack or import");
  if (m < 2 || m > 64 || m > h->max_m)
    return sgemv::report(SGEMV_ERR_ARG,
                         "sgemv_run_noalloc takes 2 <= m <= min(64, max_m) activation rows "
                         "(m = 1 needs no workspace: use sgemv_run)");
  const sgemv::Layout& L = h->L;
  if (!x_dev || !y_dev) return sgemv::report(SGEMV_ERR_ARG, "x or y is NULL");
  if ((uintptr_t)x_dev & 15u) return sgemv::report(SGEMV_ERR_ARG, "x_dev must be 16-byte aligned");
  if ((uintptr_t)y_dev & 1u) return sgemv::report(SGEMV_ERR_ARG, "y_dev must be 2-byte aligned");
  {
    const char* xb = static_cast<const char*>(x_dev);
    const char* yb = static_cast<const char*>(y_dev);
    const size_t xn = (size_t)m * L.cols * 2, yn = (size_t)m * L.rows * 2;
    if (xn && yn && xb < yb + yn && yb < xb + xn)
      return sgemv::report(SGEMV_ERR_ARG, "x and y overlap");
  }
  if (L.rows == 0) return SGEMV_OK;
  if (sgemv::tc_tiles(L) > kMaxTiles)
    return sgemv::report(SGEMV_ERR_UNSUPPORTED,
                         "rows beyond the static workspace: at most 2,097,152 weight rows "
                         "(16384 row tiles of 128)");
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return sgemv::report_cuda(e, "cudaGetDevice");
  if (prev != h->device && (e = cudaSetDevice(h->device)) != cudaSuccess)
    return sgemv::report_cuda(e, "cudaSetDevice");
  int rc = SGEMV_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  do {
    if (L.cols == 0) {
      e = cudaMemsetAsync(y_dev, 0, (size_t)m * L.rows * sizeof(__half), s);
      if (e != cudaSuccess) rc = sgemv::report_cuda(e, "zero y");
      break;
    }
    void* ws = nullptr;
    if ((e = workspace_address(h->device, &ws)) != cudaSuccess) {
      rc = sgemv::report_cuda(e, "cudaGetSymbolAddress of the static workspace");
      break;
    }
    sgemv::TcMaps maps = h->tc;   // the handle's weight maps, or encoded here (host only)
    if (!maps.ready && !sgemv::tc_encode_weights(L, h->d_vals, h->d_idx, h->d_sz, &maps)) {
      rc = sgemv::report(SGEMV_ERR_CUDA, "encoding the tensor maps of the packed weight failed");
      break;
    }
    maps.scratch = static_cast<float*>(ws);
    maps.counters = reinterpret_cast<int*>(static_cast<unsigned char*>(ws) + kPartialBytes);
    maps.ready = true;
    // the counters must start at zero (the kernel leaves them so, but the
    // array is shared with every other call and may hold an aborted call's)
    e = cudaMemsetAsync(maps.counters, 0, (size_t)sgemv::tc_tiles(L) * sizeof(int), s);
    if (e != cudaSuccess) {
      rc = sgemv::report_cuda(e, "clear the static split-K counters");
      break;
    }
    sgemv::RunArgs a;
    a.vals = h->d_vals;
    a.idx = h->d_idx;
    a.sz = h->d_sz;
    a.x = static_cast<const __half*>(x_dev);
    a.y = static_cast<__half*>(y_dev);
    a.m = m;
    a.err = h->d_err;
    e = sgemv::launch_tc(L, a, maps, s, kMaxCtas);
    if (e != cudaSuccess) rc = sgemv::report_cuda(e, "SparseGemv launch (static workspace)");
  } while (0);
  if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  return rc;
}

}  // extern "C"
