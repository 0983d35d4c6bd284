// sgemv_m1.cu -- SparseGemv for one activation row (m = 1, decode).
//
// Product (Dong et al., arXiv 2605.11582, section 1 contribution 2 and
// section 3.3): y[r] = sum over kept j of (q_j - z) * s * x[4 quad(j) + pos_j],
// fp32 accumulation, one rounding to binary16 per output.
//
// The work is bound by HBM bandwidth on the packed weight (0.81 bytes per
// kept weight), so the kernel is built around issuing few instructions per
// weight:
//
//  * Pair tables of x in shared memory.  A "pair unit" is two kept weights
//    whose columns are fixed by one 4-bit code (2:4: the quad's two
//    positions, 6 codes; 1:4: two adjacent quads' positions, 16 codes).  For
//    every unit the table holds all candidate (x_first, x_second) pairs as
//    fp32, so one 8-byte shared load fetches both activations already
//    widened.  Each lane owns a private bank column (8 bytes of every
//    128-byte line), so the data-dependent lookups never conflict.
//  * INT4 decode by the exponent trick: OR-ing a nibble shifted by p into
//    the mantissa of 2^23 gives the float 2^23 + q 2^p; subtracting
//    2^23 + z 2^p is exact and leaves (q - z) 2^p.  Five nibbles decode in
//    place, three after one shift; the 2^p factors are removed once per
//    chunk in the epilogue.
//  * Packed f32x2 arithmetic (sm_100+) for the subtract and the FMA.
//  * Each lane streams 16-byte value chunks and 8-byte index chunks with
//    non-allocating loads, kept 4 chunks ahead in a register ring, so about
//    14 KB per warp-iteration per SM are in flight.
//  * Large K is cut into slices that fit the table; row partial sums carry
//    over slices in shared memory.
//  * The weight loads of the first chunks are issued before the
//    programmatic-dependent-launch wait, so they overlap the previous
//    kernel's tail; x is read only after the wait.
#include "sgemv_internal.cuh"

namespace sgemv {
namespace {

#ifndef SGEMV_M1_NT
#define SGEMV_M1_NT 512
#endif
#ifndef SGEMV_M1_D
#define SGEMV_M1_D 2
#endif
#ifndef SGEMV_M1_MINB
#define SGEMV_M1_MINB 1
#endif
#ifndef SGEMV_M1_GRIDB
#define SGEMV_M1_GRIDB SGEMV_M1_MINB
#endif
constexpr int kNT = SGEMV_M1_NT;   // threads per CTA (one CTA per SM)
constexpr int kNW = kNT / 32;
constexpr int kD = SGEMV_M1_D;     // prefetch depth in chunks
constexpr int kSmemLimit = 227 * 1024;
constexpr uint32_t kTabAlign = 2048;
constexpr int kSmemPerSm = 228 * 1024;

template <int N>
struct M1Cfg {
  static constexpr int E = N == 2 ? 6 : 16;          // pairs per unit
  static constexpr int CPC = N == 2 ? 64 : 128;      // dense columns per chunk
  static constexpr int UC = N == 2 ? 4 : 8;          // dense columns per unit
  static constexpr int XPAD = CPC + 2;               // staged x per chunk (halves)
  // shared bytes per chunk-per-lane of slice
  static constexpr int TAB_PER_CPL = 32 * kUnitsPerChunk * E * 8;
  static constexpr int X_PER_CPL = 32 * XPAD * 2;
  static constexpr int MAX_CPL = N == 2 ? 7 : 3;
};

struct M1Params {
  const uint4* vals;
  const uint2* idx;
  const uint32_t* sz;
  const __half* x;
  __half* y;
  int rows, cols;
  int gstride;       // scale/zero words per row in memory
  int gshift;        // log2(group)
  int chunks;        // chunks holding a row's kept weights
  int cstride;       // chunks per row in memory
  int rows_per_cta;
  int slice_chunks;  // 32 * cpl
  int nslices;
  int cpl;
};

__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream8(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_nc4(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Asks the TMA unit to stage [p, p + bytes) into L2 (a hint: no data
// returns to the SM).  The range is shrunk to whole 16-byte units inside
// [lo, hi), the bounds of the buffer it belongs to.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes, const void* lo,
                                            const void* hi) {
  uintptr_t a = (uintptr_t)p, b = a + bytes;
  a = (a + 15) & ~(uintptr_t)15;
  if (a < (uintptr_t)lo) a = ((uintptr_t)lo + 15) & ~(uintptr_t)15;
  if (b > (uintptr_t)hi) b = (uintptr_t)hi;
  b &= ~(uintptr_t)15;
  while (a < b) {
    const uint32_t n = (uint32_t)min((uintptr_t)65536, b - a);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(n) : "memory");
    a += n;
  }
}

template <int OFF>
__device__ __forceinline__ float2 lds_pair(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2+%3];"
               : "=f"(v.x), "=f"(v.y)
               : "r"(addr), "n"(OFF));
  return v;
}

__device__ __forceinline__ void sts_pair(uint32_t addr, float a, float b) {
  asm volatile("st.shared.v2.f32 [%0], {%1,%2};" ::"r"(addr), "f"(a), "f"(b));
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;");
}

// Subtract constants for one (scale, zero) group: -(2^23 + z 2^p) for the
// nibble classes p = (0, 4) and (8, 12).
struct ZConst {
  float2 ca, cb;
};

__device__ __forceinline__ ZConst zconst(float z) {
  const float2 zz = make_float2(z, z);
  const float2 mm = make_float2(-8388608.0f, -8388608.0f);
  ZConst k;
  k.ca = __ffma2_rn(zz, make_float2(-1.0f, -16.0f), mm);
  k.cb = __ffma2_rn(zz, make_float2(-256.0f, -4096.0f), mm);
  return k;
}

// 2^23 + q 2^p as a float, from the nibble at bits p..p+3 of v: one LOP3
// ((v & MASK) | magic) with the exponent pattern held in a register.
template <uint32_t MASK>
__device__ __forceinline__ float mag(uint32_t v, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "n"(MASK), "r"(magic));
  return __uint_as_float(r);
}

// One 32-bit word of nibbles (pair units U0..U0+3, one per byte) times its
// x pairs.  Bytes 0 and 1 decode in place (classes 2^0,2^4 and 2^8,2^12);
// bytes 2 and 3 after a 16-bit shift, into the same classes.
template <int E, int U0, bool FIRST>
__device__ __forceinline__ void word_fma(uint32_t v, uint32_t codes, uint32_t base,
                                         uint32_t magic, const ZConst& k, float2& a0,
                                         float2& a1, float2& a2, float2& a3) {
  const uint32_t vs = v >> 16;
  float2 d0 = make_float2(mag<0xFu>(v, magic), mag<0xF0u>(v, magic));
  float2 d1 = make_float2(mag<0xF00u>(v, magic), mag<0xF000u>(v, magic));
  float2 d2 = make_float2(mag<0xFu>(vs, magic), mag<0xF0u>(vs, magic));
  float2 d3 = make_float2(mag<0xF00u>(vs, magic), mag<0xF000u>(vs, magic));
  d0 = __fadd2_rn(d0, k.ca);
  d1 = __fadd2_rn(d1, k.cb);
  d2 = __fadd2_rn(d2, k.ca);
  d3 = __fadd2_rn(d3, k.cb);
  // code of unit U0+s sits at bits 4s of `codes`; table stride 128 B/entry
  const float2 x0 = lds_pair<(U0 + 0) * E * 128>(((codes << 7) & 0x780u) | base);
  const float2 x1 = lds_pair<(U0 + 1) * E * 128>(((codes << 3) & 0x780u) | base);
  const float2 x2 = lds_pair<(U0 + 2) * E * 128>(((codes >> 1) & 0x780u) | base);
  const float2 x3 = lds_pair<(U0 + 3) * E * 128>(((codes >> 5) & 0x780u) | base);
  if (FIRST) {
    a0 = __fmul2_rn(d0, x0);
    a1 = __fmul2_rn(d1, x1);
    a2 = __fmul2_rn(d2, x2);
    a3 = __fmul2_rn(d3, x3);
  } else {
    a0 = __ffma2_rn(d0, x0, a0);
    a1 = __ffma2_rn(d1, x1, a1);
    a2 = __ffma2_rn(d2, x2, a2);
    a3 = __ffma2_rn(d3, x3, a3);
  }
}

// Removes the 2^p class factors and folds the accumulators into one float:
// a0, a2 hold classes (2^0, 2^4), a1, a3 hold (2^8, 2^12).
__device__ __forceinline__ float fold(float2 a0, float2 a1, float2 a2, float2 a3) {
  const float2 lo = __fadd2_rn(a0, a2);
  const float2 hi = __fadd2_rn(a1, a3);
  float2 t = __fmul2_rn(lo, make_float2(1.0f, 0.0625f));
  t = __ffma2_rn(hi, make_float2(0x1p-8f, 0x1p-12f), t);
  return t.x + t.y;
}

__device__ __forceinline__ float sz_scale(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float sz_zero(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// Contribution of one chunk (32 kept weights) of one row.  G2: the chunk
// spans two (scale, zero) groups (1:4 with 64-column groups), units 0..7
// in the first and 8..15 in the second.
template <int N, bool G2>
__device__ __forceinline__ float chunk_dot(const uint4& v, const uint2& ix,
                                           uint32_t sa, uint32_t sb, uint32_t base,
                                           uint32_t magic) {
  constexpr int E = M1Cfg<N>::E;
  float2 a0, a1, a2, a3;
  if (!G2) {
    const ZConst k = zconst(sz_zero(sa));
    word_fma<E, 0, true>(v.x, ix.x, base, magic, k, a0, a1, a2, a3);
    word_fma<E, 4, false>(v.y, ix.x >> 16, base, magic, k, a0, a1, a2, a3);
    word_fma<E, 8, false>(v.z, ix.y, base, magic, k, a0, a1, a2, a3);
    word_fma<E, 12, false>(v.w, ix.y >> 16, base, magic, k, a0, a1, a2, a3);
    return sz_scale(sa) * fold(a0, a1, a2, a3);
  } else {
    const ZConst ka = zconst(sz_zero(sa));
    word_fma<E, 0, true>(v.x, ix.x, base, magic, ka, a0, a1, a2, a3);
    word_fma<E, 4, false>(v.y, ix.x >> 16, base, magic, ka, a0, a1, a2, a3);
    const float ya = sz_scale(sa) * fold(a0, a1, a2, a3);
    const ZConst kb = zconst(sz_zero(sb));
    word_fma<E, 8, true>(v.z, ix.y, base, magic, kb, a0, a1, a2, a3);
    word_fma<E, 12, false>(v.w, ix.y >> 16, base, magic, kb, a0, a1, a2, a3);
    return fmaf(sz_scale(sb), fold(a0, a1, a2, a3), ya);
  }
}

// Loads of one item (the chunk a lane handles for one row).  Offsets are
// 32-bit element indices, clamped to the last element so that the zero-
// contribution items past a ragged slice or past the last row never read
// out of bounds (their table entries are zero).
template <bool G2>
struct Item {
  uint4 v;
  uint2 ix;
  uint32_t sa, sb;
  __device__ __forceinline__ void load(const M1Params& p, uint32_t o, uint32_t so,
                                       uint32_t omax, uint32_t smax) {
    o = min(o, omax);
    so = min(so, smax);
    v = ld_stream16(p.vals + o);
    ix = ld_stream8(p.idx + o);
    sa = ld_nc4(p.sz + so);
    if (G2) sb = ld_nc4(p.sz + min(so + 1, smax));
  }
};

template <int N, bool G2>
__global__ void __launch_bounds__(kNT, SGEMV_M1_MINB) k_m1(M1Params p) {
  using C = M1Cfg<N>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int S = p.cpl * kUnitsPerChunk * C::E;     // table slots per half-warp
  const int tab_bytes = 2 * S * 128;
  // The table starts on a 2 KB boundary so that bits 7..10 of every slot
  // address come from the code alone (the lookups OR the code in).
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t pad = (kTabAlign - (raw_s & (kTabAlign - 1))) & (kTabAlign - 1);
  unsigned char* tab = smem + pad;
  const uint32_t smem_s = raw_s + pad;
  __half* xs = reinterpret_cast<__half*>(tab + tab_bytes);
  float* part = reinterpret_cast<float*>(tab + tab_bytes + p.slice_chunks * C::XPAD * 2);
  const uint32_t lane_base = smem_s + (uint32_t)((lane >> 4) * S) * 128u + (lane & 15) * 8u;
  constexpr uint32_t kChunkSlotBytes = kUnitsPerChunk * C::E * 128;

  uint32_t magic = 0x4B000000u;  // exponent of 2^23, kept in a register
  asm volatile("" : "+r"(magic));
  const int r0 = blockIdx.x * p.rows_per_cta;
  const int nr = max(0, min(p.rows, r0 + p.rows_per_cta) - r0);
  const int nrw = warp < nr ? (nr - warp + kNW - 1) / kNW : 0;
  const uint32_t omax = (uint32_t)p.rows * (uint32_t)p.cstride - 1u;
  const uint32_t smax = (uint32_t)p.rows * (uint32_t)p.gstride - 1u;
  // sz index step per chunk slot (32 chunks further along the row)
  const uint32_t sstep = (uint32_t)(32 * C::CPC) >> p.gshift;

  for (int sl = 0; sl < p.nslices; ++sl) {
    const int c0 = sl * p.slice_chunks;
    const int nch = min(p.slice_chunks, p.chunks - c0);
    const int cpl = (nch + 31) >> 5;
    const int nitems = nrw * cpl;
    // load cursor: item (row j, chunk slot i) -> element offsets
    const uint32_t row0 = (uint32_t)(r0 + warp);
    uint32_t lo = row0 * (uint32_t)p.cstride + (uint32_t)(c0 + lane);
    uint32_t ls = row0 * (uint32_t)p.gstride + ((uint32_t)((c0 + lane) * C::CPC) >> p.gshift);
    const uint32_t ojump = (uint32_t)(kNW * p.cstride) - 32u * (uint32_t)(cpl - 1);
    const uint32_t sjump = (uint32_t)(kNW * p.gstride) - sstep * (uint32_t)(cpl - 1);
    int li = 0;
    auto advance = [&]() {
      const bool wrap = ++li == cpl;
      li = wrap ? 0 : li;
      lo += wrap ? ojump : 32u;
      ls += wrap ? sjump : sstep;
    };

#ifdef SGEMV_M1_L2PF
    // ---- stage this CTA's rows of the packed weight into L2 with a few
    // bulk prefetches (one contiguous range per array when K is one slice)
    if (p.nslices == 1 && threadIdx.x < 3 && nr > 0) {
      const size_t rb = (size_t)r0, re = (size_t)(r0 + nr);
      if (threadIdx.x == 0)
        prefetch_l2(p.vals + rb * p.cstride, (re - rb) * p.cstride * 16, p.vals,
                    p.vals + (size_t)p.rows * p.cstride);
      else if (threadIdx.x == 1)
        prefetch_l2(p.idx + rb * p.cstride, (re - rb) * p.cstride * 8, p.idx,
                    p.idx + (size_t)p.rows * p.cstride);
      else
        prefetch_l2(p.sz + rb * p.gstride, (re - rb) * p.gstride * 4, p.sz,
                    p.sz + (size_t)p.rows * p.gstride);
    }
#endif

    Item<G2> it[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) {
      if (d < nitems) it[d].load(p, lo, ls, omax, smax);
      advance();
    }

    if (sl == 0) {
      pdl_wait();
      pdl_launch_dependents();
    }
    __syncthreads();  // the previous slice's table is no longer read

    // ---- stage x of the slice (binary16, zero past cols), padded per chunk
    {
      const int ncols = nch * C::CPC;
      const int col0 = c0 * C::CPC;
      for (int t = threadIdx.x; t < ncols / 8; t += kNT) {
        const int col = col0 + 8 * t;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (col < p.cols) q = *reinterpret_cast<const uint4*>(p.x + col);
        const int cc = (8 * t) / C::CPC, off = (8 * t) % C::CPC;
        uint32_t* dst = reinterpret_cast<uint32_t*>(xs + cc * C::XPAD + off);
        dst[0] = q.x; dst[1] = q.y; dst[2] = q.z; dst[3] = q.w;
      }
    }
    __syncthreads();

    // ---- build the pair tables: one (lane column, chunk slot, unit) per
    // thread-iteration; a warp writes 32 different lane columns at once.
    // Slots of chunks past the slice (ragged lanes) hold zeros.
    {
      const int l = threadIdx.x & 31;
      const uint32_t colbase = smem_s + (uint32_t)((l >> 4) * S) * 128u + (l & 15) * 8u;
      for (int u_it = warp; u_it < cpl * kUnitsPerChunk; u_it += kNW) {
        const int i = u_it / kUnitsPerChunk, u = u_it % kUnitsPerChunk;
        const int cl = l + 32 * i;
        float xv[C::UC];
        if (cl < nch) {
          const __half* src = xs + cl * C::XPAD + u * C::UC;
#pragma unroll
          for (int q = 0; q < C::UC / 2; ++q) {
            const __half2 h2 = *reinterpret_cast<const __half2*>(src + 2 * q);
            xv[2 * q] = __low2float(h2);
            xv[2 * q + 1] = __high2float(h2);
          }
        } else {
#pragma unroll
          for (int q = 0; q < C::UC; ++q) xv[q] = 0.0f;
        }
        const uint32_t a = colbase + (uint32_t)(u_it * C::E) * 128u;
#pragma unroll
        for (int e = 0; e < C::E; ++e) {
          if (N == 2)
            sts_pair(a + e * 128, xv[pair24_a(e)], xv[pair24_b(e)]);
          else
            sts_pair(a + e * 128, xv[e & 3], xv[4 + (e >> 2)]);
        }
      }
    }
    __syncthreads();

    // ---- stream the rows: compute item k from ring slot k % kD, then load
    // item k + kD into that slot
    int ci = 0, cj = 0;  // (chunk slot, row) of the item being computed
    float acc = 0.0f;
    auto finish_row = [&]() {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0 && cj < nrw) {
        const int rl = warp + kNW * cj;
        if (p.nslices == 1) {
          p.y[r0 + rl] = __float2half_rn(acc);
        } else {
          const float t = (sl ? part[rl] : 0.0f) + acc;
          if (sl == p.nslices - 1)
            p.y[r0 + rl] = __float2half_rn(t);
          else
            part[rl] = t;
        }
      }
      acc = 0.0f;
      ci = 0;
      ++cj;
    };
    // Prefetches past the warp's last item read one fixed in-bounds element
    // (a cached line, no extra DRAM traffic) and are never used.
    for (int k = 0; k < nitems; k += kD) {
#pragma unroll
      for (int d = 0; d < kD; ++d) {
        if (k + d < nitems) {
          acc += chunk_dot<N, G2>(it[d].v, it[d].ix, it[d].sa, it[d].sb,
                                  lane_base + ci * kChunkSlotBytes, magic);
          const bool live = k + d + kD < nitems;
          it[d].load(p, live ? lo : omax, live ? ls : smax, omax, smax);
          advance();
          if (ci == cpl - 1) finish_row(); else ++ci;
        }
      }
    }
  }
}

int g_num_sms[64] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

template <int N, bool G2>
cudaError_t launch_m1_n(const Layout& L, const RunArgs& a, cudaStream_t s) {
  using C = M1Cfg<N>;
  const int chunks = (int)L.chunks;
  // 32-bit element offsets inside the kernel
  if ((int64_t)L.rows * L.cstride >= (1ll << 31) || (int64_t)L.rows * L.gstride >= (1ll << 31))
    return cudaErrorNotSupported;
  const int nslices = (chunks + 32 * C::MAX_CPL - 1) / (32 * C::MAX_CPL);
  const int cpl = (chunks + 32 * nslices - 1) / (32 * nslices);
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNotSupported;
  const size_t smem_body = kTabAlign + (size_t)cpl * (C::TAB_PER_CPL + C::X_PER_CPL);
  // CTAs per SM: as many as the shared memory allows, up to the launch bound
  int per_sm = SGEMV_M1_GRIDB;
  while (per_sm > 1 && smem_body * per_sm > (size_t)kSmemPerSm) --per_sm;
  int rows_per_cta = (L.rows + sms * per_sm - 1) / (sms * per_sm);
  if (nslices > 1 && rows_per_cta > 1024) rows_per_cta = 1024;
  const int grid = (L.rows + rows_per_cta - 1) / rows_per_cta;

  M1Params p;
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
  p.rows_per_cta = rows_per_cta;
  p.cpl = cpl;
  p.slice_chunks = 32 * cpl;
  p.nslices = nslices;

  const size_t smem = smem_body + (nslices > 1 ? (size_t)rows_per_cta * 4 : 0);
  if (smem > (size_t)kSmemLimit) return cudaErrorNotSupported;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_m1<N, G2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_m1<N, G2>, p);
}

}  // namespace

cudaError_t launch_m1(const Layout& L, const RunArgs& a, cudaStream_t s) {
  if (a.m != 1 || L.rows == 0 || L.cols == 0) return cudaErrorNotSupported;
  if (L.n_keep == 2) return launch_m1_n<2, false>(L, a, s);
  return L.group == 64 ? launch_m1_n<1, true>(L, a, s) : launch_m1_n<1, false>(L, a, s);
}

}  // namespace sgemv
