// sgemv_generic.cu -- the general SparseGemv kernel: any m in 1..64, either
// N, any shape.  It decodes every kept weight directly from the device
// layout and reads x through the read-only cache; the specialised kernels
// (sgemv_m1.cu) cover the hot shapes, this one covers everything else.
//
// Product (Dong et al., arXiv 2605.11582, section 1 contribution 2 and
// section 3.3): y[m][r] = sum over kept j of (q_j - z_G) * s_G * x[m][col_j],
// col_j = 4 * quad(j) + pos_j, accumulated in fp32 and rounded once to
// binary16.  (q - z) * s is exact in fp32 (a 5-bit integer times an 11-bit
// significand).
#include "sgemv_internal.cuh"

namespace sgemv {
namespace {

constexpr int kWarps = 8;
constexpr int kMTile = 8;

template <int N>
__global__ void __launch_bounds__(kWarps * 32)
k_generic(Layout L, RunArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (r >= L.rows) return;
  const uint4* vrow = a.vals + r * L.cstride;
  const uint2* irow = a.idx + r * L.cstride;
  const uint32_t* szrow = a.sz + r * L.gstride;

  for (int m0 = 0; m0 < a.m; m0 += kMTile) {
    float acc[kMTile];
#pragma unroll
    for (int i = 0; i < kMTile; ++i) acc[i] = 0.0f;

    for (int64_t c = lane; c < L.chunks; c += 32) {
      const uint4 v = vrow[c];
      const uint2 ix = irow[c];
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll 4
      for (int u = 0; u < kUnitsPerChunk; ++u) {
        const uint32_t code = ((u < 8 ? ix.x : ix.y) >> (4 * (u & 7))) & 0xFu;
        int64_t col[2];
        if (N == 2) {
          const int64_t quad = kUnitsPerChunk * c + u;
          col[0] = 4 * quad + (code & 3u);
          col[1] = 4 * quad + (code >> 2);
        } else {
          const int64_t quad = 2 * (kUnitsPerChunk * c + u);
          col[0] = 4 * quad + (code & 3u);
          col[1] = 4 * (quad + 1) + (code >> 2);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (col[h] >= L.cols) continue;   // zero-filled tail of the row
          const int i = 2 * u + h;
          const int q = (vw[i >> 3] >> (4 * (i & 7))) & 0xF;
          const uint32_t p = szrow[col[h] / L.group];
          const float s = __half2float(__ushort_as_half((unsigned short)(p & 0xFFFFu)));
          const float z = __half2float(__ushort_as_half((unsigned short)(p >> 16)));
          const float w = ((float)q - z) * s;
#pragma unroll
          for (int mm = 0; mm < kMTile; ++mm) {
            if (m0 + mm < a.m) {
              const float xv = __half2float(__ldg(a.x + (int64_t)(m0 + mm) * L.cols + col[h]));
              acc[mm] = fmaf(w, xv, acc[mm]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int mm = 0; mm < kMTile; ++mm) {
      float v = acc[mm];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && m0 + mm < a.m)
        a.y[(int64_t)(m0 + mm) * L.rows + r] = __float2half_rn(v);
    }
  }
}

}  // namespace

cudaError_t launch_generic(const Layout& L, const RunArgs& a, cudaStream_t s) {
  if (L.rows == 0 || a.m == 0) return cudaSuccess;
  const unsigned nb = (unsigned)((L.rows + kWarps - 1) / kWarps);
  if (L.n_keep == 2)
    k_generic<2><<<nb, kWarps * 32, 0, s>>>(L, a);
  else
    k_generic<1><<<nb, kWarps * 32, 0, s>>>(L, a);
  return cudaGetLastError();
}

}  // namespace sgemv
