// sgemv_format.cu -- offline format kernels: prune + quantise + pack a dense
// fp32 weight into the device layout, and convert between the device layout
// and the canonical 2bit-CSR bytes (import / export).
//
// Pruning (Dong et al., arXiv 2605.11582, section 3.2 "Sparsification",
// Eq. 3 with equal input norms and no gradient term): per quad of 4 along
// cols keep the N entries of largest |w|, ties to the lower column.
// Quantisation (section 3.2 "Adaptive group quantization"; section 1, FP16 to
// INT4): per (row, group) over the kept values, asymmetric INT4 with
// binary16 scale and zero; every float step below is a single IEEE
// operation rounded to nearest-even (explicit __f*_rn intrinsics, no
// contraction), so the result is bit-identical to any other correctly
// rounded evaluation of the same steps.
#include "sgemv_internal.cuh"

namespace sgemv {
namespace {

__device__ __forceinline__ void set_err(int* err, int code) {
  atomicCAS(err, 0, code);
}

// Keep-set of one quad: element i is kept iff fewer than N elements precede
// it in the order (larger score first, lower column first on ties).  The
// score is |w| (magnitude pruning) or the caller-weighted importance a[i].
template <int N>
__device__ __forceinline__ void prune_quad(const float w[4], const float a[4], int pos[N],
                                           float val[N]) {
  int k = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int ahead = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j != i && (a[j] > a[i] || (a[j] == a[i] && j < i))) ahead++;
    }
    if (ahead < N && k < N) {
      pos[k] = i;
      val[k] = w[i];
      ++k;
    }
  }
}

// One thread per (row, 16 dense columns).  Groups are 64..256 columns, so a
// group is 4..16 consecutive threads of one warp, reduced by xor-shuffles.
// With xnorm set, pruning ranks by the importance score of Eq. 3 (section
// 3.2): |w| * xnorm[col] + |w| * |grad| (grad NULL: zero gradient), two
// products and a sum each rounded once in binary32, as written.
template <int N>
__global__ void __launch_bounds__(256) k_pack(Layout L, RowGroups RG, int seg_max,
                                             const float* __restrict__ w,
                                             const float* __restrict__ xnorm,
                                             const float* __restrict__ grad,
                                             uint8_t* __restrict__ vals,
                                             uint8_t* __restrict__ idx,
                                             uint32_t* __restrict__ sz,
                                             int* __restrict__ err) {
  const int64_t upr = L.cols / 16;                    // units per row
  const int64_t total = (int64_t)L.rows * upr;
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = u < total;
  const int64_t r = active ? u / upr : 0;
  const int64_t k = active ? u % upr : 0;
  const int gr = RG.rowg && active ? RG.rowg[r] : L.group;   // this row's group size
  const int seg = gr / 16;                            // threads per group

  float wv[16];
  if (active) {
    const float4* src = reinterpret_cast<const float4*>(w + r * L.cols + 16 * k);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 f = src[i];
      wv[4 * i] = f.x; wv[4 * i + 1] = f.y; wv[4 * i + 2] = f.z; wv[4 * i + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = 0.0f;
  }
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) bad |= !isfinite(wv[i]);
  float sc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) sc[i] = fabsf(wv[i]);
  if (xnorm && active) {
    const float4* xs = reinterpret_cast<const float4*>(xnorm + 16 * k);
    float gv[16];
    if (grad) {
      const float4* gs = reinterpret_cast<const float4*>(grad + r * L.cols + 16 * k);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = gs[i];
        gv[4 * i] = f.x; gv[4 * i + 1] = f.y; gv[4 * i + 2] = f.z; gv[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) gv[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 n = xs[i];
      const float nv[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * i + e;
        bad |= !isfinite(gv[j]);
        sc[j] = __fadd_rn(__fmul_rn(sc[j], nv[e]), __fmul_rn(sc[j], fabsf(gv[j])));
      }
    }
  }
  if (bad) set_err(err, kDevErrNonfinite);

  int pos[4][N];
  float val[4][N];
  float lo = 0.0f, hi = 0.0f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    prune_quad<N>(&wv[4 * t], &sc[4 * t], pos[t], val[t]);
#pragma unroll
    for (int n = 0; n < N; ++n) {
      lo = fminf(lo, val[t][n]);
      hi = fmaxf(hi, val[t][n]);
    }
  }
  // groups are seg-aligned runs of lanes (a row's units start at a multiple
  // of cols/16, a multiple of seg); every lane joins every shuffle and keeps
  // only partners of its own group
  for (int off = 1; off < seg_max; off <<= 1) {
    const float olo = __shfl_xor_sync(0xffffffffu, lo, off);
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
    if (off < seg) {
      lo = fminf(lo, olo);
      hi = fmaxf(hi, ohi);
    }
  }
  if (!active || bad) return;

  unsigned short s16;
  int z;
  if (hi == lo) {
    s16 = 0x3C00u;
    z = 0;
  } else {
    const float range = __fsub_rn(hi, lo);
    if (!isfinite(range)) { set_err(err, kDevErrRange); return; }
    s16 = __half_as_ushort(__float2half_rn(__fdiv_rn(range, 15.0f)));
    if ((s16 & 0x7FFFu) == 0x7C00u) { set_err(err, kDevErrRange); return; }
    if (s16 == 0) s16 = 1;
    const float sf = __half2float(__ushort_as_half(s16));
    float zf = rintf(__fdiv_rn(-lo, sf));
    zf = fminf(fmaxf(zf, 0.0f), 15.0f);
    z = (int)zf;
  }
  const float sf = __half2float(__ushort_as_half(s16));
  const float zfl = (float)z;

  int q[4][N];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
#pragma unroll
    for (int n = 0; n < N; ++n) {
      float qf = __fadd_rn(rintf(__fdiv_rn(val[t][n], sf)), zfl);
      qf = fminf(fmaxf(qf, 0.0f), 15.0f);
      q[t][n] = (int)qf;
    }
  }

  // Device layout: the row's kept weights are contiguous, 32 per 16-byte
  // chunk, in canonical nibble order.  This thread owns kept weights
  // [4N k, 4N (k+1)) of the row.
  const int64_t vrow = L.cstride * 16;  // device bytes per row (vals)
  const int64_t irow = L.cstride * 8;   // device bytes per row (idx)
  if constexpr (N == 2) {
    uint32_t vw = 0;
    uint32_t iw = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      vw |= (uint32_t)(q[t][0] | (q[t][1] << 4)) << (8 * t);
      iw |= (uint32_t)(pos[t][0] | (pos[t][1] << 2)) << (4 * t);
    }
    *reinterpret_cast<uint32_t*>(vals + r * vrow + 4 * k) = vw;
    *reinterpret_cast<uint16_t*>(idx + r * irow + 2 * k) = (uint16_t)iw;
  } else {
    uint32_t vw = 0;
    uint32_t iw = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      vw |= (uint32_t)q[t][0] << (4 * t);
      iw |= (uint32_t)pos[t][0] << (2 * t);
    }
    *reinterpret_cast<uint16_t*>(vals + r * vrow + 2 * k) = (uint16_t)vw;
    idx[r * irow + k] = (uint8_t)iw;
  }
  // the thread at the start of each device group (L.group columns; a row's
  // coarser group covers several) writes the group's scale and zero there
  if ((16 * k) % L.group == 0) {
    const unsigned short z16 = __half_as_ushort(__float2half_rn(zfl));
    sz[r * L.gstride + (16 * k) / L.group] = (uint32_t)s16 | ((uint32_t)z16 << 16);
  }
}

// Canonical -> device: one thread per (row, chunk slot in memory); slots
// past the row's kept weights are written as zeros.
template <int N>
__global__ void k_canon_to_device(Layout L, const uint8_t* __restrict__ cvals,
                                  const uint8_t* __restrict__ cidx,
                                  uint8_t* __restrict__ vals,
                                  uint8_t* __restrict__ idx,
                                  int* __restrict__ err) {
  const int64_t total = (int64_t)L.rows * L.cstride;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int64_t r = t / L.cstride, c = t % L.cstride;
  const uint8_t* vsrc = cvals + r * L.vals_row;
  const uint8_t* isrc = cidx + r * L.idx_row;
  uint8_t* vdst = vals + (r * L.cstride + c) * 16;
  uint8_t* idst = idx + (r * L.cstride + c) * 8;
  for (int b = 0; b < 16; ++b) {
    const int64_t o = 16 * c + b;
    vdst[b] = o < L.vals_row ? vsrc[o] : 0;
  }
  for (int b = 0; b < 8; ++b) {
    const int64_t o = 8 * c + b;
    uint8_t byte = o < L.idx_row ? isrc[o] : 0;
    if constexpr (N == 2) {
      // two quads per byte, (a | b << 2) in each nibble; the positions must
      // ascend (a rejected byte becomes positions (0, 1), and pack fails)
      if (o < L.idx_row) {
        for (int h = 0; h < 2; ++h) {
          const int nib = (byte >> (4 * h)) & 0xF;
          if ((nib & 3) >= (nib >> 2)) {
            set_err(err, kDevErrBadIndex);
            byte = (uint8_t)((byte & ~(0xF << (4 * h))) | (0x4 << (4 * h)));
          }
        }
      } else {
        byte = 0x44;   // padding chunk: zero codes at positions (0, 1)
      }
    }
    idst[b] = byte;
  }
}

// One thread per (row, device group of L.group columns).  The canonical
// entry of device group Gd of row r is its row group Gd * L.group / g_r.
__global__ void k_sz_to_device(Layout L, RowGroups RG, const uint16_t* __restrict__ scale,
                               const uint16_t* __restrict__ zero,
                               uint32_t* __restrict__ sz) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)L.rows * L.ngroups) return;
  const int64_t r = i / L.ngroups, Gd = i % L.ngroups;
  const int gr = RG.rowg ? RG.rowg[r] : L.group;
  const int64_t ci = (RG.goff ? RG.goff[r] : r * L.ngroups) + Gd * L.group / gr;
  sz[r * L.gstride + Gd] = (uint32_t)scale[ci] | ((uint32_t)zero[ci] << 16);
}

__global__ void k_sz_to_canon(Layout L, RowGroups RG, const uint32_t* __restrict__ sz,
                              uint16_t* __restrict__ scale,
                              uint16_t* __restrict__ zero) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)L.rows * L.ngroups) return;
  const int64_t r = i / L.ngroups, Gd = i % L.ngroups;
  const int gr = RG.rowg ? RG.rowg[r] : L.group;
  if ((Gd * L.group) % gr != 0) return;   // not the first sub-slot of its row group
  const int64_t ci = (RG.goff ? RG.goff[r] : r * L.ngroups) + Gd * L.group / gr;
  const uint32_t w = sz[r * L.gstride + Gd];
  scale[ci] = (uint16_t)(w & 0xFFFFu);
  zero[ci] = (uint16_t)(w >> 16);
}

// Device -> canonical: one thread per (row, chunk).
template <int N>
__global__ void k_device_to_canon(Layout L, const uint8_t* __restrict__ vals,
                                  const uint8_t* __restrict__ idx,
                                  uint8_t* __restrict__ cvals,
                                  uint8_t* __restrict__ cidx) {
  const int64_t total = (int64_t)L.rows * L.chunks;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int64_t r = t / L.chunks, c = t % L.chunks;
  const uint8_t* vsrc = vals + (r * L.cstride + c) * 16;
  const uint8_t* isrc = idx + (r * L.cstride + c) * 8;
  uint8_t* vdst = cvals + r * L.vals_row;
  uint8_t* idst = cidx + r * L.idx_row;
  for (int b = 0; b < 16; ++b) {
    const int64_t o = 16 * c + b;
    if (o < L.vals_row) vdst[o] = vsrc[b];
  }
  for (int b = 0; b < 8; ++b) {
    const int64_t o = 8 * c + b;
    if (o >= L.idx_row) continue;
    idst[o] = isrc[b];
  }
}

inline unsigned blocks_for(int64_t n, int threads) {
  return (unsigned)((n + threads - 1) / threads);
}

}  // namespace

cudaError_t launch_pack(const Layout& L, const RowGroups& G, const float* w, const float* xnorm,
                        const float* grad, uint4* vals, uint2* idx, uint32_t* sz, int* err,
                        cudaStream_t s) {
  const int64_t total = (int64_t)L.rows * (L.cols / 16);
  if (total == 0) return cudaSuccess;
  const unsigned nb = blocks_for(total, 256);
  const int seg_max = G.rowg ? 16 : L.group / 16;
  if (L.n_keep == 2)
    k_pack<2><<<nb, 256, 0, s>>>(L, G, seg_max, w, xnorm, grad, reinterpret_cast<uint8_t*>(vals),
                                 reinterpret_cast<uint8_t*>(idx), sz, err);
  else
    k_pack<1><<<nb, 256, 0, s>>>(L, G, seg_max, w, xnorm, grad, reinterpret_cast<uint8_t*>(vals),
                                 reinterpret_cast<uint8_t*>(idx), sz, err);
  return cudaGetLastError();
}

cudaError_t launch_canon_to_device(const Layout& L, const RowGroups& G, const uint8_t* cvals,
                                   const uint8_t* cidx, const uint16_t* scale,
                                   const uint16_t* zero, uint4* vals, uint2* idx,
                                   uint32_t* sz, int* err, cudaStream_t s) {
  const int64_t total = (int64_t)L.rows * L.cstride;
  if (total > 0) {
    if (L.n_keep == 2)
      k_canon_to_device<2><<<blocks_for(total, 256), 256, 0, s>>>(
          L, cvals, cidx, reinterpret_cast<uint8_t*>(vals),
          reinterpret_cast<uint8_t*>(idx), err);
    else
      k_canon_to_device<1><<<blocks_for(total, 256), 256, 0, s>>>(
          L, cvals, cidx, reinterpret_cast<uint8_t*>(vals),
          reinterpret_cast<uint8_t*>(idx), err);
  }
  const int64_t ns = (int64_t)L.rows * L.ngroups;
  if (ns > 0) k_sz_to_device<<<blocks_for(ns, 256), 256, 0, s>>>(L, G, scale, zero, sz);
  return cudaGetLastError();
}

cudaError_t launch_device_to_canon(const Layout& L, const RowGroups& G, const uint4* vals,
                                   const uint2* idx, const uint32_t* sz,
                                   uint8_t* cvals, uint8_t* cidx, uint16_t* scale,
                                   uint16_t* zero, cudaStream_t s) {
  const int64_t total = (int64_t)L.rows * L.chunks;
  if (total > 0) {
    if (L.n_keep == 2)
      k_device_to_canon<2><<<blocks_for(total, 256), 256, 0, s>>>(
          L, reinterpret_cast<const uint8_t*>(vals),
          reinterpret_cast<const uint8_t*>(idx), cvals, cidx);
    else
      k_device_to_canon<1><<<blocks_for(total, 256), 256, 0, s>>>(
          L, reinterpret_cast<const uint8_t*>(vals),
          reinterpret_cast<const uint8_t*>(idx), cvals, cidx);
  }
  const int64_t ns = (int64_t)L.rows * L.ngroups;
  if (ns > 0) k_sz_to_canon<<<blocks_for(ns, 256), 256, 0, s>>>(L, G, sz, scale, zero);
  return cudaGetLastError();
}

}  // namespace sgemv
