// sgemv_mma.cu -- SparseGemv for a small batch of activation rows on the
// tensor cores with the warp-level sparse MMA: 2 <= m <= 32 (beam
// candidates / prefix-tree verification nodes; larger batches run the
// tcgen05 kernel of sgemv_tc.cu, and this kernel takes any m <= 64), 2:4
// weights and 1:4 weights (each kept weight paired with a zero).
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
//  * metadata: the stored position nibbles (a | b << 2) are the MMA's own
//    format; thread (g, t in {0,1}) supplies quads 4t..4t+3 of rows g (low
//    half) and g + 8 (high half), one PRMT of the two rows' code words.
//  * B (32 x 8): x rows staged in shared memory (padded rows, so ldmatrix
//    reads are conflict-free), one ldmatrix.x4 per n-tile and k-tile.
//  * weights and x: the CTA's 128 rows x K sub-slice (codes, positions and
//    the sub-slice's scale/zero words) and the sub-slice's x columns are
//    copied into shared memory with cp.async, double-buffered across equal
//    sub-slices, as few as fit; the first sub-slice's weights are in flight
//    before the wait for the previous kernel.  Warps read their rows from
//    padded rows of the buffer (conflict-free).
//  * scale: each k-tile lies inside one group; the MMA accumulates a group
//    into a temporary that is scaled by s and added in fp32.
//  * split-K across the CTAs of a thread-block cluster, reduced through
//    distributed shared memory in rank order -- deterministic, no global
//    scratch.  With one n-tile (m <= 8) every CTA pushes its partial rows
//    to their owner rank with remote stores counted on the owner's mbarrier
//    (one split cluster barrier, arrive at launch and wait after the main
//    loop, orders the setup); wider tiles are written to each CTA's shared
//    memory and pulled by the owners between two cluster barriers.
#include <string.h>

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
#ifndef SGEMV_MMA_CPS
#define SGEMV_MMA_CPS 2
#endif
constexpr int kCtasPerSm = SGEMV_MMA_CPS;   // CTAs resident per SM
constexpr size_t kSmemPerCta = (kCtasPerSm == 1 ? 227 : 113) * 1024;
// Shared-memory buffers (weights + x) of the sub-slice ring.  Two: three or
// four, with as many smaller sub-slices, measured 2-11 us slower per layer
// step at m = 4..16.
#ifndef SGEMV_MMA_STAGES
#define SGEMV_MMA_STAGES 2
#endif
constexpr int kStages = SGEMV_MMA_STAGES;
static_assert(kStages >= 2 && kStages <= 6, "sub-slice ring: 2..6 buffers");
// Sub-slices per CTA the planner aims for (at least; smaller ones when the
// shared memory needs it)
// Chunk loop of the main loop unrolled by two: the next chunk's shared
// loads and decode overlap this one's MMAs (layer steps 0.4-2 us faster at
// m = 4..24; by four: no further gain)
#ifndef SGEMV_MMA_CUNROLL
#define SGEMV_MMA_CUNROLL 2
#endif
constexpr int kChunkUnroll = SGEMV_MMA_CUNROLL;
#ifndef SGEMV_MMA_GCHUNK
#define SGEMV_MMA_GCHUNK 1
#endif
constexpr bool kGroupPerChunk = SGEMV_MMA_GCHUNK != 0;
#ifndef SGEMV_MMA_PULL4
#define SGEMV_MMA_PULL4 1
#endif
constexpr bool kPullVec4 = SGEMV_MMA_PULL4 != 0;
#ifndef SGEMV_MMA_NSUB_MIN
#define SGEMV_MMA_NSUB_MIN 1
#endif
#ifndef SGEMV_MMA_PDL
#define SGEMV_MMA_PDL 1
#endif

// One packed matrix of a launch: a launch covers up to kMaxSegs matrices
// that share x, cols and N; their 128-row tiles are numbered in order.
constexpr int kMaxSegs = 8;
struct MmaSeg {
  const uint4* vals;
  const uint2* idx;
  const uint32_t* sz;
  __half* y;
  int rows, gstride, gshift, ngroups;
  int tile_begin;     // first row tile of this matrix in the launch
};

struct MmaParams {
  MmaSeg seg[kMaxSegs];
  int nseg;
  // the CTA's matrix (copied from seg[] at the start of the kernel)
  const uint4* vals;
  const uint2* idx;
  const uint32_t* sz;
  const __half* x;
  __half* y;
  int rows, cols, gstride, gshift, chunks, cstride;
  int m;
  int split_chunks;   // chunks per cluster rank
  int nsplit;         // cluster size
  int sub_chunks;     // chunks of weights and x staged at a time
  int sub_groups;     // scale/zero words per row staged per sub-slice (bound)
  int ngroups;        // scale/zero groups per row
  int row_tile0;      // (the CTA's matrix) its first tile in the launch
  int* err;           // device error word (a bounded wait that gave up)
  // Failure-detection test hook (0 in normal use): every rank withholds its
  // split-K partials, so each owner's bounded wait runs out after wait_ns.
  int withhold;
  unsigned long long wait_ns;   // the owner's wait limit
};

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

template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src) {
  if (BYTES == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(BYTES)
                 : "memory");
}
// 16 bytes, of which the first `src_bytes` (0 or 16) come from src and the
// rest are zero
__device__ __forceinline__ void cp_async_zfill(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// ---- cluster reduction primitives: an mbarrier counting the bytes that the
// other ranks push, their remote stores, and the split cluster barrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, float a, float b, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
      "f"(a), "f"(b), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void sts_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// A wait gives up after this long (ns): far beyond any legitimate stall.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
// The limit under the failure-detection test hook (the bytes never come).
constexpr unsigned long long kInjectWaitNs = 20000ull;

// The split-K partials travel by remote stores from the accumulators (one
// 8-byte store per row pair and n-tile, counted on the owner's mbarrier) for
// one n-tile; wider tiles write them to shared memory and the owners pull
// them after a cluster barrier.  At two n-tiles the pulled form measured
// 1-3 us faster per layer step (the pushed one issues 1024 remote stores per
// CTA); at one n-tile the two forms time the same.
#ifndef SGEMV_MMA_PUSH_NT
#define SGEMV_MMA_PUSH_NT 1
#endif
__host__ __device__ constexpr bool push_reduce(int nt) { return nt <= SGEMV_MMA_PUSH_NT; }

// Rows of the CTA tile that cluster rank q reduces: [q R / n, (q + 1) R / n).
__device__ __forceinline__ int owner_rank(int r, int nsplit) {
  return ((r + 1) * nsplit - 1) / kRowsCta;
}

// 1:4 operand of quads t and t + 4 of k-step kt for one row, as two half2
// MMA registers.  Each kept weight is paired with a zero at the other
// position of its half of the quad -- positions (0, 1) for a < 2, (2, 3)
// otherwise -- so the 2:4 sparse MMA computes exactly its product; the
// value sits in the low half for even a and the high half for odd a.  w is
// vals word kt (quads 8kt .. 8kt + 7, one code per nibble); pw the
// positions shifted so that quad t's are bits 0..1 and quad t + 4's bits
// 8..9; z1024 = (1024 + z, 1024 + z).
__device__ __forceinline__ void quads14(uint32_t w, int t, uint32_t pw, uint32_t z1024,
                                        uint32_t& r_t, uint32_t& r_t4) {
  uint32_t h;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(h) : "r"(w >> (4 * t)));
  uint32_t v;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(v) : "r"(h), "r"(z1024));   // (v_t, v_t4)
  r_t = __byte_perm(v, 0u, 0x4410u - (pw & 1u) * 0x33CCu);
  r_t4 = __byte_perm(v, 0u, 0x4432u - ((pw >> 8) & 1u) * 0x11EEu);
}

// 1:4 metadata of MMA quads 4t'..4t'+3 (t' = t % 2): e holds the position
// byte of those quads for row g (bits 0..7) and row g + 8 (bits 16..23).
// A position a selects the pair (0, 1) when a < 2 and (2, 3) otherwise:
// nibble 4 or 14 -- 4 | 10 h with h the high bit of a.
__device__ __forceinline__ uint32_t meta14(uint32_t e) {
  e &= 0x00AA00AAu;                                          // h at bits 1, 3, 5, 7
  uint32_t x = (e & 0x000A000Au) | ((e & 0x00A000A0u) << 4); // -> 1, 3, 9, 11
  x = (x & 0x02020202u) | ((x & 0x08080808u) << 2);          // -> 1, 5, 9, 13
  return x | (x << 2) | 0x44444444u;
}

// (scale as float, (1024 + z, 64 + z) as half2) of one (row, group).
__device__ __forceinline__ void group_consts(uint32_t szw, float& s, uint32_t& zc) {
  s = __half2float(__ushort_as_half((unsigned short)(szw & 0xFFFFu)));
  const uint32_t zz = __byte_perm(szw, 0u, 0x3232u);  // (z, z)
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(zc) : "r"(zz), "r"(0x54006400u));
}

// Shared-memory geometry of one weight buffer: the CTA's 128 rows x SC
// chunks of a K sub-slice.  Row strides are padded by one element so that
// the 8 rows a warp instruction reads fall in different banks.
struct WGeom {
  int sc;        // chunks per sub-slice
  int gs;        // scale/zero words per row and sub-slice (upper bound)
  int vst, ist, sst;          // row strides in bytes
  int vals_off, idx_off, sz_off, bytes;
  __host__ __device__ WGeom(int sc_, int gs_) : sc(sc_), gs(gs_) {
    vst = sc * 16 + 16;
    ist = sc * 8 + 8;
    sst = (gs + 1) * 4;
    vals_off = 0;
    idx_off = kRowsCta * vst;
    sz_off = idx_off + kRowsCta * ist;
    bytes = (sz_off + kRowsCta * sst + 127) & ~127;
  }
};

// (row, column) of a thread's pieces in an R x n block walked in steps of
// the CTA size: one division at the start, then carries.
struct Walk2D {
  int r, c, dr, dc, n;
  __device__ __forceinline__ Walk2D(int n_) : n(n_) {
    r = (int)threadIdx.x / n;
    c = (int)threadIdx.x - r * n;
    dr = (kW * 32) / n;
    dc = (kW * 32) - dr * n;
  }
  __device__ __forceinline__ void step() {
    c += dc;
    r += dr;
    if (c >= n) {
      c -= n;
      ++r;
    }
  }
};

// Copies the weight block of rows [row0, row0 + 128) x chunks [cs, ce) and
// the scale/zero words of groups [g0, g1] into a buffer; rows past the
// matrix are skipped (their values are replaced when read).
__device__ __forceinline__ void stage_weights(const MmaParams& p, const WGeom& W, uint32_t buf,
                                              int row0, int cs, int ce, int g0, int g1) {
  const int nc = ce - cs, ng = g1 - g0 + 1;
  const int nrow = min(kRowsCta, p.rows - row0);
  for (Walk2D w(nc); w.r < nrow; w.step()) {
    const size_t src = (size_t)(row0 + w.r) * p.cstride + cs + w.c;
    cp_async<16>(buf + W.vals_off + w.r * W.vst + w.c * 16, p.vals + src);
    cp_async<8>(buf + W.idx_off + w.r * W.ist + w.c * 8, p.idx + src);
  }
  for (Walk2D w(ng); w.r < nrow; w.step())
    cp_async<4>(buf + W.sz_off + w.r * W.sst + w.c * 4,
                p.sz + (size_t)(row0 + w.r) * p.gstride + g0 + w.c);
}

template <int NT, int N>
__global__ void __launch_bounds__(kW * 32, kCtasPerSm) k_mma24(const __grid_constant__ MmaParams pp) {
  constexpr int CPC = N == 2 ? 64 : 128;   // dense columns per chunk
  constexpr int KT = CPC / 32;             // MMA k-steps per chunk
  extern __shared__ __align__(128) unsigned char smem[];
  MmaParams p = pp;   // scalars; the CTA's matrix is filled in below
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int mp = NT * 8;                       // padded activation rows
  const int xs_stride = p.sub_chunks * CPC + 8; // halves per staged x row
  const WGeom W(p.sub_chunks, p.sub_groups);
  // shared memory: x of kStages sub-slices | kStages weight buffers |
  // (pushed reduction) the receive buffer, one slot of ceil(R / nsplit) rows
  // x mp per rank, and its mbarrier.  Sub-slice s uses x and weight buffer
  // s % kStages.  The pulled reduction writes its partial tile over the
  // front once the main loop is done.
  const uint32_t xs_s = (uint32_t)__cvta_generic_to_shared(smem);
  const int xs_bytes = (mp * xs_stride * 2 + 127) & ~127;
  const uint32_t wbuf0 = xs_s + (uint32_t)(kStages * xs_bytes);
  float* part = reinterpret_cast<float*>(smem);
  const int rq = (kRowsCta + p.nsplit - 1) / p.nsplit;
  const uint32_t recv_s = wbuf0 + (uint32_t)(kStages * W.bytes);
  const uint32_t rbar = recv_s + (uint32_t)(p.nsplit * rq * mp * 4);
  const float* recv = reinterpret_cast<const float*>(smem + (recv_s - xs_s));

  // the matrix of this CTA's row tile
  const int tile = (int)blockIdx.x / p.nsplit;
  {
    int si = 0;
    while (si + 1 < pp.nseg && tile >= pp.seg[si + 1].tile_begin) ++si;
    const MmaSeg& sg = pp.seg[si];
    p.vals = sg.vals;
    p.idx = sg.idx;
    p.sz = sg.sz;
    p.y = sg.y;
    p.rows = sg.rows;
    p.gstride = sg.gstride;
    p.gshift = sg.gshift;
    p.ngroups = sg.ngroups;
    p.row_tile0 = sg.tile_begin;
  }
  const int row0 = (tile - p.row_tile0) * kRowsCta;
  const int rowbase = row0 + warp * 16;
  const int rg = rowbase + g, rg8 = rowbase + g + 8;
  const bool vg = rg < p.rows, vg8 = rg8 < p.rows;
  const int lr_g = warp * 16 + g, lr_g8 = lr_g + 8;   // rows within the CTA
  const int c_begin = rank * p.split_chunks;
  const int c_end = min(p.chunks, c_begin + p.split_chunks);
  const int nsub = c_end > c_begin ? (c_end - c_begin + p.sub_chunks - 1) / p.sub_chunks : 0;

  float acc[NT][4];
  float tmp[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[n][i] = tmp[n][i] = 0.0f;

  // selectors copying byte t (or t + 4 of the word pair) into bytes 0 and 2
  const uint32_t sel = 0x4040u | (uint32_t)t | ((uint32_t)t << 8);
  // ... and the 16-bit metadata field of thread t from rows g, g + 8
  const uint32_t msel = (t & 1) ? 0x7632u : 0x5410u;
  float s_g = 0.0f, s_g8 = 0.0f;
  uint32_t zc_g = 0, zc_g8 = 0;
  int cur_group = -1;

  // ldmatrix row address of this thread: matrix j = lane / 8, row lane % 8
  const uint32_t ld_base = xs_s + (uint32_t)(((lane & 7) * xs_stride + (lane >> 3) * 8) * 2);

  // this rank's rows of the reduction; the bytes the other ranks will push
  const int r_lo = rank * kRowsCta / p.nsplit, r_hi = (rank + 1) * kRowsCta / p.nsplit;
  if constexpr (push_reduce(NT)) {
    if (threadIdx.x == 0) {
      mbar_init(rbar, 1);
      mbar_arrive_expect_tx(rbar, (uint32_t)((p.nsplit - 1) * (r_hi - r_lo) * mp * 4));
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // first half of a cluster barrier: every rank's receive side is set up
    // before any rank pushes (the wait comes after the main loop)
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  }

  // x[:, CPC cs .. CPC ce) into x buffer xb, zero for padded rows (cols is a
  // multiple of the group, so no 16-byte piece crosses the end of a row)
  auto stage_x = [&](uint32_t xb, int cs, int ce) {
    for (Walk2D w((ce - cs) * (CPC / 8)); w.r < mp; w.step()) {
      const int col = cs * CPC + w.c * 8;
      const bool in = w.r < p.m && col < p.cols;
      cp_async_zfill(xb + (uint32_t)((w.r * xs_stride + w.c * 8) * 2),
                     in ? p.x + (size_t)w.r * p.cols + col : p.x, in ? 16 : 0);
    }
  };
  // weights of the first kStages - 1 sub-slices: in flight while the
  // previous kernel ends (one commit group)
  for (int sp = 0; sp < kStages - 1 && sp < nsub; ++sp) {
    const int cs = c_begin + sp * p.sub_chunks, ce = min(c_end, cs + p.sub_chunks);
    stage_weights(p, W, wbuf0 + (uint32_t)(sp * W.bytes), row0, cs, ce, (cs * CPC) >> p.gshift,
                  min(p.ngroups - 1, (ce * CPC - 1) >> p.gshift));
  }
  cp_commit();
  // x may be written by the previous kernel: wait for it only now; one
  // commit group per sub-slice's x
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  for (int sp = 0; sp < kStages - 1; ++sp) {
    if (sp < nsub) {
      const int cs = c_begin + sp * p.sub_chunks;
      stage_x(xs_s + (uint32_t)(sp * xs_bytes), cs, min(c_end, cs + p.sub_chunks));
    }
    cp_commit();
  }

  // Ring of kStages buffers: sub-slice i sits in buffer i % kStages; while
  // one is computed the next kStages - 1 are in flight.  Every iteration
  // commits one group, so "sub-slice sidx landed" is always "at most
  // kStages - 1 groups pending".
  for (int sidx = 0; sidx < nsub; ++sidx) {
    const int cs = c_begin + sidx * p.sub_chunks;
    const int ce = min(c_end, cs + p.sub_chunks);
    const int g0 = (cs * CPC) >> p.gshift;
    const int bi = sidx % kStages;
    const uint32_t wb = wbuf0 + (uint32_t)(bi * W.bytes);
    const uint32_t ld_x = ld_base + (uint32_t)(bi * xs_bytes);
    __syncthreads();  // previous sub-slice fully consumed: its buffers are free
    if (sidx + kStages - 1 < nsub) {
      // sub-slice sidx + kStages - 1 into the buffers sub-slice sidx - 1 used
      const int ns = c_begin + (sidx + kStages - 1) * p.sub_chunks;
      const int ne = min(c_end, ns + p.sub_chunks);
      const int nb = (sidx + kStages - 1) % kStages;
      stage_weights(p, W, wbuf0 + (uint32_t)(nb * W.bytes), row0, ns, ne,
                    (ns * CPC) >> p.gshift, min(p.ngroups - 1, (ne * CPC - 1) >> p.gshift));
      stage_x(xs_s + (uint32_t)(nb * xs_bytes), ns, ne);
    }
    cp_commit();
    cp_wait<kStages - 1>();   // this thread's copies of sub-slice sidx landed
    __syncthreads();          // ... and every thread's
#pragma unroll kChunkUnroll
    for (int c = cs; c < ce; ++c) {
      const int cc = c - cs;
      uint4 v_g = make_uint4(0, 0, 0, 0), v_g8 = v_g;
      uint2 i_g = make_uint2(0, 0), i_g8 = i_g;
      if (vg) {
        v_g = lds128(wb + W.vals_off + lr_g * W.vst + cc * 16);
        i_g = lds64(wb + W.idx_off + lr_g * W.ist + cc * 8);
      }
      if (vg8) {
        v_g8 = lds128(wb + W.vals_off + lr_g8 * W.vst + cc * 16);
        i_g8 = lds64(wb + W.idx_off + lr_g8 * W.ist + cc * 8);
      }
      if constexpr (kChecked && N == 2) {
        if ((vg && (bad_codes24(i_g.x) | bad_codes24(i_g.y))) ||
            (vg8 && (bad_codes24(i_g8.x) | bad_codes24(i_g8.y)))) {
          report_checked(p.err);
          if (vg) i_g = make_uint2(0x44444444u, 0x44444444u);
          if (vg8) i_g8 = make_uint2(0x44444444u, 0x44444444u);
        }
      }
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        if (N == 1 && c * CPC + kt * 32 >= p.cols) break;   // ragged 1:4 tail
        int G = (c * CPC + kt * 32) >> p.gshift;
        // 2:4 chunks are 64 columns and groups at least as wide: only a
        // chunk's first k-step can open a group
        if ((N == 1 || kt == 0 || !kGroupPerChunk) && G != cur_group) {
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
          if constexpr (kChecked) {
            if (G - g0 < 0 || G - g0 >= W.gs) {
              report_checked(p.err);
              G = g0;
            }
          }
          const uint32_t w_g = vg ? lds32(wb + W.sz_off + lr_g * W.sst + (G - g0) * 4) : 0x3C00u;
          const uint32_t w_g8 = vg8 ? lds32(wb + W.sz_off + lr_g8 * W.sst + (G - g0) * 4) : 0x3C00u;
          group_consts(w_g, s_g, zc_g);
          group_consts(w_g8, s_g8, zc_g8);
        }
        uint32_t a0, a1, a2, a3, meta;
        if constexpr (N == 2) {
          const uint32_t wlo_g = kt ? v_g.z : v_g.x, whi_g = kt ? v_g.w : v_g.y;
          const uint32_t wlo_g8 = kt ? v_g8.z : v_g8.x, whi_g8 = kt ? v_g8.w : v_g8.y;
          a0 = quad_h2(wlo_g, sel, zc_g);    // row g,   quad t
          a1 = quad_h2(wlo_g8, sel, zc_g8);  // row g+8, quad t
          a2 = quad_h2(whi_g, sel, zc_g);    // row g,   quad t+4
          a3 = quad_h2(whi_g8, sel, zc_g8);  // row g+8, quad t+4
          // metadata (threads t = 0, 1): the stored position nibbles of quads
          // 4t..4t+3 of this k-tile, row g in the low half, row g+8 in the high
          meta = __byte_perm(kt ? i_g.y : i_g.x, kt ? i_g8.y : i_g8.x, msel);
        } else {
          // quads 8kt + t and 8kt + t + 4: vals word kt, positions in idx word
          // kt / 2 from bit 16 (kt % 2) + 2t
          const uint32_t w_g = kt == 0 ? v_g.x : kt == 1 ? v_g.y : kt == 2 ? v_g.z : v_g.w;
          const uint32_t w_g8 = kt == 0 ? v_g8.x : kt == 1 ? v_g8.y : kt == 2 ? v_g8.z : v_g8.w;
          const uint32_t iw_g = kt < 2 ? i_g.x : i_g.y, iw_g8 = kt < 2 ? i_g8.x : i_g8.y;
          const int sh = 16 * (kt & 1) + 2 * t;
          // (1024 + z) in both halves: the high half of zc is 64 + z
          const uint32_t z1024_g = __byte_perm(zc_g, 0u, 0x1010u);
          const uint32_t z1024_g8 = __byte_perm(zc_g8, 0u, 0x1010u);
          quads14(w_g, t, iw_g >> sh, z1024_g, a0, a2);
          quads14(w_g8, t, iw_g8 >> sh, z1024_g8, a1, a3);
          const uint32_t bi = 2 * (kt & 1) + (t & 1);   // position byte of quads 4t'..4t'+3
          meta = meta14(__byte_perm(iw_g, iw_g8, bi | (bi << 4) | ((4 + bi) << 8) | ((4 + bi) << 12)));
        }
        const uint32_t kofs = (uint32_t)((cc * CPC + kt * 32) * 2);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(ld_x + (uint32_t)(n * 8 * xs_stride * 2) + kofs, b0, b1, b2, b3);
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
  cp_wait<0>();

  if constexpr (!push_reduce(NT)) {
    // ---- split-K reduction across the cluster, pulled (rank order,
    // deterministic): every CTA writes its fp32 partial tile to its own
    // shared memory; each rank reads its rows from all ranks
    __syncthreads();  // every warp is done with x and the buffers: part reuses them
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int mc = n * 8 + 2 * t;
      part[lr_g * mp + mc] = acc[n][0];
      part[lr_g * mp + mc + 1] = acc[n][1];
      part[lr_g8 * mp + mc] = acc[n][2];
      part[lr_g8 * mp + mc + 1] = acc[n][3];
    }
    cluster.sync();
    if (kPullVec4) {
      // four activation rows per load: 16-byte loads from every rank's
      // partial tile (rows of mp floats, mp a multiple of 8), all ranks'
      // loads in flight together, summed in rank order
      const int nq = mp / 4;
      const int n_el = (r_hi - r_lo) * nq;
      const uint32_t part_s = (uint32_t)__cvta_generic_to_shared(part);
      uint32_t rb[kMaxSplit];
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q) rb[q] = map_rank(part_s, q < p.nsplit ? q : 0);
      for (int e = threadIdx.x; e < n_el; e += kW * 32) {
        const int lr = r_lo + e / nq, m4 = (e % nq) * 4;
        const uint32_t off = (uint32_t)((lr * mp + m4) * 4);
        float4 v[kMaxSplit];
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
          v[q] = q < p.nsplit ? ld_cluster_f4(rb[q] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
        float sx = 0.0f, sy = 0.0f, sz = 0.0f, sw = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q) {
          sx += v[q].x;
          sy += v[q].y;
          sz += v[q].z;
          sw += v[q].w;
        }
        const int row = row0 + lr;
        if (row < p.rows) {
          __half* yr = p.y + row;
          if (m4 < p.m) yr[(size_t)m4 * p.rows] = __float2half_rn(sx);
          if (m4 + 1 < p.m) yr[(size_t)(m4 + 1) * p.rows] = __float2half_rn(sy);
          if (m4 + 2 < p.m) yr[(size_t)(m4 + 2) * p.rows] = __float2half_rn(sz);
          if (m4 + 3 < p.m) yr[(size_t)(m4 + 3) * p.rows] = __float2half_rn(sw);
        }
      }
    } else {
      const int n_el = (r_hi - r_lo) * p.m;
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
    return;
  }

  // ---- split-K reduction across the cluster, pushed (rank order,
  // deterministic): every rank sends its partial rows to the rank that owns
  // them straight from the accumulators (remote stores counted on the
  // owner's mbarrier); an owner sums the nsplit slots of its rows in rank
  // order
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = h ? lr_g8 : lr_g;
    const int q = owner_rank(r, p.nsplit);
    const int rl = r - q * kRowsCta / p.nsplit;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const uint32_t off = (uint32_t)(((rank * rq + rl) * mp + n * 8 + 2 * t) * 4);
      const float a = acc[n][2 * h], b = acc[n][2 * h + 1];
      if (q == rank)
        sts_v2(recv_s + off, a, b);
      else if (!p.withhold)
        st_async_v2(map_rank(recv_s + off, q), a, b, map_rank(rbar, q));
    }
  }
  // second split cluster barrier: this rank's sends are issued; no CTA
  // leaves before every rank has issued its own, so no remote store can
  // target a CTA that has retired
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  __syncthreads();  // this rank's own slot is in place
  // The owner's wait for the other ranks' bytes is bounded: with a byte
  // count that can never be reached it records SGEMV_ERR_TIMEOUT and skips
  // the sum instead of spinning forever.
  bool ok = mbar_try_wait(rbar, 0);
  if (!ok) {
    const unsigned long long t0 = global_ns();
    while (!(ok = mbar_try_wait(rbar, 0)))
      if (global_ns() - t0 > p.wait_ns) break;
  }
  const bool timed_out = __syncthreads_or(!ok) != 0;   // one decision per CTA
  if (!timed_out) {
    const int n_el = (r_hi - r_lo) * p.m;
    for (int e = threadIdx.x; e < n_el; e += kW * 32) {
      const int rl = e / p.m, mm = e % p.m;
      float sum = 0.0f;
      for (int q = 0; q < p.nsplit; ++q) sum += recv[(q * rq + rl) * mp + mm];
      const int row = row0 + r_lo + rl;
      if (row < p.rows) p.y[(size_t)mm * p.rows + row] = __float2half_rn(sum);
    }
  } else if (threadIdx.x == 0) {
    atomicCAS(p.err, 0, kDevErrTimeout);
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (timed_out) {
    // every rank's sends are issued by now: give stores still in flight a
    // bounded time to land before this CTA's shared memory is released
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(rbar, 0))
      if (global_ns() - t0 > p.wait_ns) break;
  }
}

// Shared memory of a launch with sub-slices of `sc` chunks of `cpc` columns.
size_t mma_smem(int nt, int sc, int group, int cpc, int nsplit) {
  const int mp = nt * 8;
  const WGeom W(sc, (sc * cpc + group - 1) / group + 1);
  const size_t xs = ((size_t)mp * (sc * cpc + 8) * 2 + 127) & ~(size_t)127;
  const size_t main = (size_t)kStages * (xs + (size_t)W.bytes);
  if (!push_reduce(nt)) {
    const size_t red = (size_t)kRowsCta * mp * 4;
    return main > red ? main : red;
  }
  const size_t recv = (size_t)nsplit * ((kRowsCta + nsplit - 1) / nsplit) * mp * 4;
  return main + recv + 16;
}

// One launch over `count` matrices that share x, cols, N and m.
template <int NT, int N>
cudaError_t launch_nt(const Layout* Ls, const RunArgs* as, int count, cudaStream_t s, int sms) {
  constexpr int CPC = N == 2 ? 64 : 128;
  const Layout& L0 = Ls[0];
  const RunArgs& a = as[0];
  const int chunks = (int)L0.chunks;
  int ntiles = 0, gmin = 256;
  MmaParams p;
  memset(&p, 0, sizeof p);
  for (int i = 0; i < count; ++i) {
    MmaSeg& sg = p.seg[i];
    sg.vals = as[i].vals;
    sg.idx = as[i].idx;
    sg.sz = as[i].sz;
    sg.y = as[i].y;
    sg.rows = Ls[i].rows;
    sg.gstride = (int)Ls[i].gstride;
    sg.gshift = Ls[i].group == 64 ? 6 : (Ls[i].group == 128 ? 7 : 8);
    sg.ngroups = (int)Ls[i].ngroups;
    sg.tile_begin = ntiles;
    ntiles += (Ls[i].rows + kRowsCta - 1) / kRowsCta;
    gmin = min(gmin, Ls[i].group);
  }
  for (int i = count; i < kMaxSegs; ++i) p.seg[i].tile_begin = ntiles;
  p.nseg = count;
  if (ntiles == 0) return cudaSuccess;
  // as many K splits as keep every CTA resident in one wave
  int nsplit = (kCtasPerSm * sms) / ntiles;
  nsplit = max(1, min(kMaxSplit, min(nsplit, chunks)));
  const int split_chunks = (chunks + nsplit - 1) / nsplit;
  nsplit = (chunks + split_chunks - 1) / split_chunks;
  // sub-slices of equal size, as few as fit two CTAs per SM (the smallest
  // group has the most scale/zero words per sub-slice); each costs two CTA
  // barriers and a pipeline fill, and more, smaller ones measured slower
  int nsb = max(1, min(SGEMV_MMA_NSUB_MIN, split_chunks));
  int sub = min(64, (split_chunks + nsb - 1) / nsb);
  while (sub > 1 && mma_smem(NT, sub, gmin, CPC, nsplit) > kSmemPerCta) {
    ++nsb;
    sub = (split_chunks + nsb - 1) / nsb;
  }
  const size_t smem = mma_smem(NT, sub, gmin, CPC, nsplit);
  if (smem > 227 * 1024) return cudaErrorNotSupported;
  p.x = a.x;
  p.cols = L0.cols;
  p.cstride = (int)L0.cstride;
  p.chunks = chunks;
  p.m = a.m;
  p.split_chunks = split_chunks;
  p.nsplit = nsplit;
  p.sub_chunks = sub;
  p.sub_groups = (sub * CPC + gmin - 1) / gmin + 1;
  p.err = a.err;
  p.withhold = a.withhold;
  p.wait_ns = a.withhold ? kInjectWaitNs : kWaitLimitNs;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_mma24<NT, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    if (kMaxSplit > 8) {
      e = cudaFuncSetAttribute(k_mma24<NT, N>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles * nsplit);
  cfg.blockDim = dim3(kW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = SGEMV_MMA_PDL ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_mma24<NT, N>, p);
}

int g_sms[64] = {0};

}  // namespace

bool withhold_applies(const Layout& L, int m) {
  // one n-tile: this kernel's pushed split-K sums; m > mma_max_m(N): the
  // tcgen05 kernel's x copies.  The pulled sums of wider tiles wait on
  // cluster barriers only, which every rank reaches: nothing to withhold.
  const bool pushed = push_reduce((m + 7) / 8);
  return m >= 2 && (pushed || m > mma_max_m(L.n_keep)) && L.rows > 0 && L.cols > 0;
}

cudaError_t launch_mma_group(const Layout* Ls, const RunArgs* as, int count, cudaStream_t s) {
  if (count < 1 || count > kMaxSegs) return cudaErrorNotSupported;
  const int m = as[0].m;
  for (int i = 0; i < count; ++i)
    if (as[i].m != m || Ls[i].cols != Ls[0].cols || Ls[i].n_keep != Ls[0].n_keep ||
        Ls[i].rows == 0 || Ls[i].cols == 0)
      return cudaErrorNotSupported;
  if (m < 2 || m > 64) return cudaErrorNotSupported;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorNotSupported;
    g_sms[dev] = n;
  }
  const int nt = (m + 7) / 8;
  const int sms = g_sms[dev];
  if (count > 1) {
    int ntiles = 0;
    for (int i = 0; i < count; ++i) ntiles += (Ls[i].rows + kRowsCta - 1) / kRowsCta;
    if (kCtasPerSm * sms / ntiles < 2) {
      // one launch could not split K: each CTA would walk a whole row of
      // sub-slices; separate launches, each split, measured faster
      for (int i = 0; i < count; ++i) {
        const cudaError_t e = launch_mma_group(Ls + i, as + i, 1, s);
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
  }
  if (Ls[0].n_keep == 2) {
    switch (nt) {
      case 1: return launch_nt<1, 2>(Ls, as, count, s, sms);
      case 2: return launch_nt<2, 2>(Ls, as, count, s, sms);
      case 3: return launch_nt<3, 2>(Ls, as, count, s, sms);
      case 4: return launch_nt<4, 2>(Ls, as, count, s, sms);
      case 5: return launch_nt<5, 2>(Ls, as, count, s, sms);
      case 6: return launch_nt<6, 2>(Ls, as, count, s, sms);
      case 7: return launch_nt<7, 2>(Ls, as, count, s, sms);
      default: return launch_nt<8, 2>(Ls, as, count, s, sms);
    }
  }
  switch (nt) {
    case 1: return launch_nt<1, 1>(Ls, as, count, s, sms);
    case 2: return launch_nt<2, 1>(Ls, as, count, s, sms);
    case 3: return launch_nt<3, 1>(Ls, as, count, s, sms);
    case 4: return launch_nt<4, 1>(Ls, as, count, s, sms);
    case 5: return launch_nt<5, 1>(Ls, as, count, s, sms);
    case 6: return launch_nt<6, 1>(Ls, as, count, s, sms);
    case 7: return launch_nt<7, 1>(Ls, as, count, s, sms);
    default: return launch_nt<8, 1>(Ls, as, count, s, sms);
  }
}

cudaError_t launch_mma(const Layout& L, const RunArgs& a, cudaStream_t s) {
  if (a.m < 2 || a.m > 64 || L.rows == 0 || L.cols == 0)
    return cudaErrorNotSupported;
  return launch_mma_group(&L, &a, 1, s);
}

}  // namespace sgemv
