// sgemv_mma.cu -- SparseGemv for a small batch of activation rows on the
// tensor cores: 2:4 weights, 2 <= m <= 64 (beam candidates / prefix-tree
// verification nodes).
//
// Product (Dong et al., arXiv 2605.11582, section 1 contribution 2 and
// section 3.3, applied to the verification batch of section 3.1):
//   y[m][r] = sum_G s_rG * sum_{kept j in G} (q_j - z_rG) * x[m][col_j],
// fp32 accumulation, binary16 output.
//
// The 2:4 sparse MMA (mma.sp, m16n8k32, f16 inputs, f32 accumulation) takes
// the compressed weight tile plus 2-bit in-quad positions as metadata --
// exactly what a 2bit-CSR quad stores -- so no dense expansion happens:
//  * A (16 rows x 32 dense columns, 16 kept per row): (q - z) decoded to
//    binary16 in registers.  One PRMT copies a quad's byte (two nibbles) to
//    both halves, one LOP3 keeps q_a in the low half's mantissa and q_b in
//    the high half's (exponent patterns for 1024 and 64), one HSUB2 takes
//    (1024 + z, 64 + z) off.  (q - z) is an integer in [-15, 15], exact.
//  * metadata: the stored six-way pair codes become (a | b << 2) nibbles
//    through a PRMT lookup table; thread (g, t in {0,1}) supplies quads
//    4t..4t+3 of rows g (low half) and g + 8 (high half).
//  * B (32 x 8): x rows staged in shared memory (padded rows, so ldmatrix
//    reads are conflict-free), one ldmatrix.x4 per n-tile and k-tile.
//  * scale: each k-tile lies inside one group; the MMA accumulates a group
//    into a temporary that is scaled by s and added in fp32.
//  * split-K across the CTAs of a thread-block cluster: every CTA writes its
//    fp32 partial tile to its own shared memory and the cluster reduces the
//    tile through distributed shared memory in rank order -- deterministic,
//    no global scratch.
#include <cooperative_groups.h>

#include "sgemv_internal.cuh"

namespace cg = cooperative_groups;

namespace sgemv {
namespace {

constexpr int kW = 8;                 // warps per CTA
constexpr int kRowsCta = 16 * kW;     // weight rows per CTA
#ifndef SGEMV_MMA_MAXSPLIT
#define SGEMV_MMA_MAXSPLIT 8
#endif
constexpr int kMaxSplit = SGEMV_MMA_MAXSPLIT;  // CTAs per cluster (portable limit 8)
constexpr int kXBudget = 64 * 1024;   // bytes of staged x per CTA

struct MmaParams {
  const uint4* vals;
  const uint2* idx;
  const uint32_t* sz;
  const __half* x;
  __half* y;
  int rows, cols, gstride, gshift, chunks, cstride;
  int m;
  int split_chunks;   // chunks per cluster rank
  int nsplit;         // cluster size
  int sub_chunks;     // chunks of x staged at a time
};

// code (0..5) -> (a | b << 2): (0,1)=4 (0,2)=8 (0,3)=12 (1,2)=9 (1,3)=13 (2,3)=14
constexpr uint32_t kMetaLo = 0x090C0804u;
constexpr uint32_t kMetaHi = 0x00000E0Du;

// Four stored codes (a 16-bit field) -> four metadata nibbles (16 bits).
__device__ __forceinline__ uint32_t meta16(uint32_t codes) {
  uint32_t r = __byte_perm(kMetaLo, kMetaHi, codes & 0xFFFFu);
  r |= r >> 4;
  return __byte_perm(r, 0u, 0x4420u);
}

// half2 (q_a - z, q_b - z) of the quad whose byte is byte `t` of `w`.
__device__ __forceinline__ uint32_t quad_h2(uint32_t w, uint32_t sel, uint32_t zc) {
  uint32_t r = __byte_perm(w, 0u, sel);
  asm("lop3.b32 %0, %1, 0x00F0000F, 0x54006400, 0xEA;" : "=r"(r) : "r"(r));
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(r), "r"(zc));
  return d;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_sp(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1, uint32_t b2,
                                       uint32_t b3, uint32_t meta) {
  asm volatile(
      "mma.sp::ordered_metadata.sync.aligned.m16n8k32.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, 0x0;"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(b2), "r"(b3),
        "r"(meta));
}

__device__ __forceinline__ uint4 ld_nc16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_nc8(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// (scale as float, (1024 + z, 64 + z) as half2) of one (row, group).
__device__ __forceinline__ void group_consts(uint32_t szw, float& s, uint32_t& zc) {
  s = __half2float(__ushort_as_half((unsigned short)(szw & 0xFFFFu)));
  const uint32_t zz = __byte_perm(szw, 0u, 0x3232u);  // (z, z)
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(zc) : "r"(zz), "r"(0x54006400u));
}

template <int NT>
__global__ void __launch_bounds__(kW * 32, 2) k_mma24(MmaParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int mp = NT * 8;                       // padded activation rows
  const int xs_stride = p.sub_chunks * 64 + 8; // halves per staged x row
  __half* xs = reinterpret_cast<__half*>(smem);
  float* part = reinterpret_cast<float*>(smem + (size_t)mp * xs_stride * 2);
  const uint32_t xs_s = (uint32_t)__cvta_generic_to_shared(xs);

  const int rowbase = (blockIdx.x / p.nsplit) * kRowsCta + warp * 16;
  const int rg = rowbase + g, rg8 = rowbase + g + 8;
  const bool vg = rg < p.rows, vg8 = rg8 < p.rows;
  const int c_begin = rank * p.split_chunks;
  const int c_end = min(p.chunks, c_begin + p.split_chunks);

  float acc[NT][4];
  float tmp[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[n][i] = tmp[n][i] = 0.0f;

  // selectors copying byte t (or t + 4 of the word pair) into bytes 0 and 2
  const uint32_t sel = 0x4040u | (uint32_t)t | ((uint32_t)t << 8);
  float s_g = 0.0f, s_g8 = 0.0f;
  uint32_t zc_g = 0, zc_g8 = 0;
  int cur_group = -1;

  // ldmatrix row address of this thread: matrix j = lane / 8, row lane % 8
  const uint32_t ld_base = xs_s + (uint32_t)(((lane & 7) * xs_stride + (lane >> 3) * 8) * 2);

  for (int cs = c_begin; cs < c_end; cs += p.sub_chunks) {
    const int ce = min(c_end, cs + p.sub_chunks);
    __syncthreads();  // previous sub-slice fully consumed
    {
      // stage x[:, 64 cs .. 64 ce) (zero for padded rows)
      const int ncol = (ce - cs) * 64;
      const int pieces = mp * (ncol / 8);
      for (int i = threadIdx.x; i < pieces; i += kW * 32) {
        const int row = i / (ncol / 8), c8 = i % (ncol / 8);
        uint4 q = make_uint4(0, 0, 0, 0);
        if (row < p.m)
          q = *reinterpret_cast<const uint4*>(p.x + (size_t)row * p.cols + cs * 64 + c8 * 8);
        *reinterpret_cast<uint4*>(xs + row * xs_stride + c8 * 8) = q;
      }
    }
    __syncthreads();
    for (int c = cs; c < ce; ++c) {
      uint4 v_g = make_uint4(0, 0, 0, 0), v_g8 = v_g;
      uint2 i_g = make_uint2(0, 0), i_g8 = i_g;
      if (vg) {
        v_g = ld_nc16(p.vals + (size_t)rg * p.cstride + c);
        i_g = ld_nc8(p.idx + (size_t)rg * p.cstride + c);
      }
      if (vg8) {
        v_g8 = ld_nc16(p.vals + (size_t)rg8 * p.cstride + c);
        i_g8 = ld_nc8(p.idx + (size_t)rg8 * p.cstride + c);
      }
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        const int G = (c * 64 + kt * 32) >> p.gshift;
        if (G != cur_group) {
          if (cur_group >= 0) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              acc[n][0] = fmaf(s_g, tmp[n][0], acc[n][0]);
              acc[n][1] = fmaf(s_g, tmp[n][1], acc[n][1]);
              acc[n][2] = fmaf(s_g8, tmp[n][2], acc[n][2]);
              acc[n][3] = fmaf(s_g8, tmp[n][3], acc[n][3]);
              tmp[n][0] = tmp[n][1] = tmp[n][2] = tmp[n][3] = 0.0f;
            }
          }
          cur_group = G;
          const uint32_t w_g = vg ? p.sz[(size_t)rg * p.gstride + G] : 0x3C00u;
          const uint32_t w_g8 = vg8 ? p.sz[(size_t)rg8 * p.gstride + G] : 0x3C00u;
          group_consts(w_g, s_g, zc_g);
          group_consts(w_g8, s_g8, zc_g8);
        }
        const uint32_t wlo_g = kt ? v_g.z : v_g.x, whi_g = kt ? v_g.w : v_g.y;
        const uint32_t wlo_g8 = kt ? v_g8.z : v_g8.x, whi_g8 = kt ? v_g8.w : v_g8.y;
        const uint32_t a0 = quad_h2(wlo_g, sel, zc_g);    // row g,   quad t
        const uint32_t a1 = quad_h2(wlo_g8, sel, zc_g8);  // row g+8, quad t
        const uint32_t a2 = quad_h2(whi_g, sel, zc_g);    // row g,   quad t+4
        const uint32_t a3 = quad_h2(whi_g8, sel, zc_g8);  // row g+8, quad t+4
        // metadata (threads t = 0, 1): quads 4t..4t+3 of rows g and g+8
        const uint32_t cw_g = kt ? i_g.y : i_g.x, cw_g8 = kt ? i_g8.y : i_g8.x;
        const uint32_t sh = (t & 1) * 16;
        const uint32_t meta = meta16(cw_g >> sh) | (meta16(cw_g8 >> sh) << 16);
        const uint32_t kofs = (uint32_t)(((c - cs) * 64 + kt * 32) * 2);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(ld_base + (uint32_t)(n * 8 * xs_stride * 2) + kofs, b0, b1, b2, b3);
          mma_sp(tmp[n], a0, a1, a2, a3, b0, b1, b2, b3, meta);
        }
      }
    }
  }
  if (cur_group >= 0) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      acc[n][0] = fmaf(s_g, tmp[n][0], acc[n][0]);
      acc[n][1] = fmaf(s_g, tmp[n][1], acc[n][1]);
      acc[n][2] = fmaf(s_g8, tmp[n][2], acc[n][2]);
      acc[n][3] = fmaf(s_g8, tmp[n][3], acc[n][3]);
    }
  }

  // ---- split-K reduction across the cluster (rank order, deterministic)
  // part: [kRowsCta][mp] fp32 of this CTA
  const int lr_g = warp * 16 + g, lr_g8 = lr_g + 8;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int mc = n * 8 + 2 * t;
    part[lr_g * mp + mc] = acc[n][0];
    part[lr_g * mp + mc + 1] = acc[n][1];
    part[lr_g8 * mp + mc] = acc[n][2];
    part[lr_g8 * mp + mc + 1] = acc[n][3];
  }
  cluster.sync();
  {
    // rank k finishes rows [k * kRowsCta / nsplit, (k+1) * kRowsCta / nsplit)
    const int r_lo = rank * kRowsCta / p.nsplit, r_hi = (rank + 1) * kRowsCta / p.nsplit;
    const int n_el = (r_hi - r_lo) * p.m;
    const int row0 = (blockIdx.x / p.nsplit) * kRowsCta;
    const float* rp[kMaxSplit];
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q)
      rp[q] = cluster.map_shared_rank(part, q < p.nsplit ? q : 0);
    for (int e = threadIdx.x; e < n_el; e += kW * 32) {
      const int lr = r_lo + e / p.m, mm = e % p.m;
      float v[kMaxSplit];
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q) v[q] = q < p.nsplit ? rp[q][lr * mp + mm] : 0.0f;
      float sum = 0.0f;
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q) sum += v[q];
      const int row = row0 + lr;
      if (row < p.rows) p.y[(size_t)mm * p.rows + row] = __float2half_rn(sum);
    }
  }
  cluster.sync();  // no CTA leaves while its partial tile is being read
}

template <int NT>
cudaError_t launch_nt(const Layout& L, const RunArgs& a, cudaStream_t s, int sms) {
  const int chunks = (int)L.chunks;
  const int ntiles = (L.rows + kRowsCta - 1) / kRowsCta;
#ifndef SGEMV_MMA_CTAS_PER_SM
#define SGEMV_MMA_CTAS_PER_SM 2
#endif
  int nsplit = (SGEMV_MMA_CTAS_PER_SM * sms + ntiles - 1) / ntiles;
  nsplit = max(1, min(kMaxSplit, min(nsplit, chunks)));
  const int split_chunks = (chunks + nsplit - 1) / nsplit;
  nsplit = (chunks + split_chunks - 1) / split_chunks;
  // x staged per sub-slice: mp rows x (64 sub + 8) halves within budget
  const int mp = NT * 8;
  int sub = (kXBudget / (mp * 2) - 8) / 64;
  sub = max(1, min(sub, split_chunks));
  MmaParams p;
  p.vals = a.vals;
  p.idx = a.idx;
  p.sz = a.sz;
  p.x = a.x;
  p.y = a.y;
  p.rows = L.rows;
  p.cols = L.cols;
  p.gstride = (int)L.gstride;
  p.cstride = (int)L.cstride;
  p.gshift = L.group == 64 ? 6 : (L.group == 128 ? 7 : 8);
  p.chunks = chunks;
  p.m = a.m;
  p.split_chunks = split_chunks;
  p.nsplit = nsplit;
  p.sub_chunks = sub;
  const size_t smem = (size_t)mp * (sub * 64 + 8) * 2 + (size_t)kRowsCta * mp * 4;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_mma24<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    if (kMaxSplit > 8) {
      e = cudaFuncSetAttribute(k_mma24<NT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles * nsplit);
  cfg.blockDim = dim3(kW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_mma24<NT>, p);
}

int g_sms[64] = {0};

}  // namespace

cudaError_t launch_mma(const Layout& L, const RunArgs& a, cudaStream_t s) {
  if (L.n_keep != 2 || a.m < 2 || a.m > 64 || L.rows == 0 || L.cols == 0)
    return cudaErrorNotSupported;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorNotSupported;
    g_sms[dev] = n;
  }
  const int nt = (a.m + 7) / 8;
  switch (nt) {
    case 1: return launch_nt<1>(L, a, s, g_sms[dev]);
    case 2: return launch_nt<2>(L, a, s, g_sms[dev]);
    case 3: return launch_nt<3>(L, a, s, g_sms[dev]);
    case 4: return launch_nt<4>(L, a, s, g_sms[dev]);
    case 5: return launch_nt<5>(L, a, s, g_sms[dev]);
    case 6: return launch_nt<6>(L, a, s, g_sms[dev]);
    case 7: return launch_nt<7>(L, a, s, g_sms[dev]);
    default: return launch_nt<8>(L, a, s, g_sms[dev]);
  }
}

}  // namespace sgemv
