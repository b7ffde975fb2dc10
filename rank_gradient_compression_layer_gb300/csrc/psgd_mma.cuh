// The project phase for padded ranks 16 and 32 on the tensor cores (tcgen05).
//
// At r >= 16 the project tile's arithmetic outgrows its bytes: per element
// and worker, the error rebuild E = B - Phat' Q_w'^T is r multiply-adds, and
// the CUDA-core kernel is bound by feeding those from shared memory.  Here
// the rebuild is a tensor-core product per (tile, worker):
//
//   D_w^T (128 columns x 128 rows, TMEM) = Q_w'_segment (128 x r) Phat'_tile^T
//
// in error-compensated TF32 (hi/lo split, three MMAs per K step: float32
// accuracy), and the tile's share of P is one more product after the
// workers, P_tile (128 x r) = Msum (128 x 128) Q_segment (128 x r), with
// Msum = sum_w M_w (P is linear in M).  D is formed transposed so that a
// TMEM lane is a column: each thread takes its column's D values straight
// from its lane, streams G and B of that column (a warp covers 32
// consecutive columns: 128-byte rows), forms M_w = G_w + (B_w - D_w),
// stores it to B_w and adds it to Msum.
//
// A CTA owns 128 rows x one segment (128 columns, the TMEM lanes) and loops
// over the workers; worker w + 1's Q_w' rows are staged and its MMAs issued
// while worker w's rows are combined (D in two TMEM buffers).  G and B come
// into shared memory by 16-byte asynchronous copies (cp.async.cg: 512 bytes
// per warp request), a ring of NS chunks per row quarter (8 rows x the
// segment's columns of G and of B), NS - 1 chunks ahead across the workers;
// each thread then reads its own column from the chunk.  Every wait on the
// tensor cores is bounded; one that runs out marks the step's status word
// (the host reports it) and the tile is abandoned.
#pragma once

#include "psgd_kernels.cuh"
#include "psgd_umma.cuh"

namespace psgd {

constexpr int kMThreads = 512;    // 16 warps: 4 TMEM lane groups (columns) x 4 row quarters
constexpr int kMRows = 128;       // rows of a tile
constexpr int kMCols = kSeg * 4;  // columns of a tile (one segment): the TMEM lanes of D

template <int RP>
struct MmaCfg {
  static_assert(RP == 16 || RP == 32, "tensor-core project tiles are for padded ranks 16 and 32");
  static constexpr uint32_t OP = (uint32_t)kMRows * RP * 4;     // one copy (hi or lo) of a 128 x r operand
  static constexpr uint32_t MS = (uint32_t)kMRows * kMCols * 4;  // one copy of Msum
  static constexpr uint32_t OFF_P = 0;                          // Phat' tile hi, lo; later the P rows, Gram scratch
  static constexpr uint32_t OFF_Q = 2 * OP;                     // Q^T hi, lo (the P product's B operand)
  static constexpr uint32_t OFF_U = OFF_Q + 2 * OP;             // Q_w' buffers 0, 1 (hi, lo each), then Msum hi, lo
  // Msum as the P product's A operand (128 rows x K = 128 columns, K-major):
  // its K-adjacent core matrices 144 bytes apart, 16 more than packed, so that
  // a warp's stores of one row's 32 columns hit 32 distinct banks
  static constexpr uint32_t M_LBO = 144;
  static constexpr uint32_t M_SBO = (kMCols / 4) * M_LBO;
  static constexpr uint32_t MS_P = (kMRows / 8) * M_SBO;  // one copy of the padded Msum
  static constexpr uint32_t U_BYTES = (4 * OP > 2 * MS_P) ? 4 * OP : 2 * MS_P;
  // the rings, after the Q_w' buffers, over Msum's space (Msum is formed
  // after the worker loop): 4 row quarters x NS chunks of 8 rows x 128
  // columns of G and of B, as many chunks as fit
  static constexpr uint32_t CHUNK = 2u * 8 * kMCols * 4;
  static constexpr uint32_t OFF_R = OFF_U + 4 * OP;
  static constexpr int NS = (int)((227u * 1024 - 1024 - OFF_R) / (4 * CHUNK)) < 5
                                ? (int)((227u * 1024 - 1024 - OFF_R) / (4 * CHUNK))
                                : 5;
  static_assert(NS >= 2, "a ring of at least two chunks");
  static constexpr uint32_t RING = 4u * NS * CHUNK;
  static constexpr uint32_t SMEM = (OFF_U + U_BYTES > OFF_R + RING) ? OFF_U + U_BYTES : OFF_R + RING;
  static_assert(SMEM <= 227 * 1024, "fits the shared memory of one CTA");
  static constexpr uint32_t TMEM_COLS = 512;  // D of two workers (2 x 128) and the P tile (r)
  static_assert((uint32_t)kMRows * RP * 4 + RP * RP * 8 <= 2 * OP, "P rows and Gram scratch fit over the Phat' tile");
  static_assert(kMRows <= Cfg<RP>::R1MAX, "the split step's Gram tile holds a whole row block");
};

// Stages a rows x RP row-major float32 block (rows past `valid`, or all when
// `zero`, as zeros) as the hi and lo copies of a K-major operand, K = RP.
template <int RP>
__device__ __forceinline__ void stage_kmajor_rows(unsigned char* hi, unsigned char* lo, const float* src, int rows,
                                                  int valid, bool zero) {
  constexpr int K4 = RP / 4;
  for (int e = threadIdx.x; e < rows * K4; e += blockDim.x) {
    const int r = e / K4, k4 = e - r * K4;
    float4 v = zero4();
    if (!zero && r < valid) v = __ldg(reinterpret_cast<const float4*>(src + (int64_t)r * RP) + k4);
    float4 h, l;
    tf32_split(v.x, h.x, l.x);
    tf32_split(v.y, h.y, l.y);
    tf32_split(v.z, h.z, l.z);
    tf32_split(v.w, h.w, l.w);
    const uint32_t o = umma_off(r, 4 * k4, RP);
    *reinterpret_cast<float4*>(hi + o) = h;
    *reinterpret_cast<float4*>(lo + o) = l;
  }
}

// One project tile: 128 rows x one segment, all workers.  D_w is formed
// transposed, D_w^T (128 columns x 128 rows) = Q_w'_seg Phat'_tile^T, so
// that TMEM lane = column: thread (lane group g = warp % 4, row quarter
// q = warp / 4) owns column 32 g + lane and rows 32 q .. 32 q + 31, reads
// its D values straight from its lane, and its G and B accesses are
// 128-byte rows per warp.
template <int RP>
__global__ void __launch_bounds__(kMThreads, 1) p1m_kernel(const StepArgs a) {
  using C = MmaCfg<RP>;
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t s_mbar[3];
  __shared__ uint32_t s_tmem;
  __shared__ int s_flag;
  pdl_enter();
  const Tile t = a.tiles[blockIdx.x];
  const LayerDev L = a.layers[t.layer];  // by value: stores to B cannot alias it
  const P1Tile T = p1_tile<RP>(a, t, L);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cl = 32 * (warp & 3) + lane;  // this thread's column in the segment (its TMEM lane)
  const int r0 = 32 * (warp >> 2);        // its first row in the tile
  const int col = T.seg * kMCols + cl;    // column in the layer
  const bool col_in = col < L.ld;         // inside the row (padding included)
  const int segcols = min(kMCols, L.ld - T.seg * kMCols);
  const bool prev = T.prev;
  const uint32_t base = smem_u32(sm);

  if (warp == 0) tmem_alloc(&s_tmem, C::TMEM_COLS);
  if (tid == 0) {
    mbar_init(&s_mbar[0]);
    mbar_init(&s_mbar[1]);
    mbar_init(&s_mbar[2]);
  }
  if (prev)
    stage_kmajor_rows<RP>(sm + C::OFF_P, sm + C::OFF_P + C::OP, a.Phat + L.p_off + (int64_t)T.row0 * RP, kMRows,
                          T.rcnt, false);
  auto stage_qw = [&](int w) {
    unsigned char* buf = sm + C::OFF_U + (uint32_t)(w & 1) * 2 * C::OP;
    stage_kmajor_rows<RP>(buf, buf + C::OP, a.Qw + (int64_t)w * a.q_total + L.q_off + (int64_t)T.seg * kMCols * RP,
                          kMCols, segcols, false);
  };
  if (prev) stage_qw(0);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  // D_w^T = Q_w' Phat'^T into TMEM columns (w & 1) * 128: hi hi + hi lo + lo hi
  auto issue_e = [&](int w) {
    constexpr uint32_t id = umma_idesc_tf32(kMCols, kMRows);
    const uint32_t d = tmem + (uint32_t)(w & 1) * kMRows;
    const uint32_t ahi = base + C::OFF_U + (uint32_t)(w & 1) * 2 * C::OP, alo = ahi + C::OP;
    const uint32_t bhi = base + C::OFF_P, blo = bhi + C::OP;
#pragma unroll 1
    for (int ks = 0; ks < RP / 8; ++ks) {
      const uint32_t o = (uint32_t)ks * 256;
      umma_tf32(d, umma_sdesc(ahi + o, RP), umma_sdesc(bhi + o, RP), id, ks > 0 ? 1u : 0u);
      umma_tf32(d, umma_sdesc(ahi + o, RP), umma_sdesc(blo + o, RP), id, 1u);
      umma_tf32(d, umma_sdesc(alo + o, RP), umma_sdesc(bhi + o, RP), id, 1u);
    }
    umma_commit(&s_mbar[w & 1]);
  };
  if (prev && tid == 0) issue_e(0);

  float msum[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) msum[i] = 0.f;
  // Item i = chunk i % 4 (rows r0 + 8 (i % 4) .. + 7) of worker i / 4, in
  // slot i % NS of this row quarter's ring: G rows [8][128] floats, then B
  // rows.  The quarter's 128 threads copy it together (2 float4 of G and 2 of
  // B each); thread (column cl) reads its column.
  const int q = warp >> 2, jq = tid & 127;  // row quarter, thread within it
  const int n_items = 4 * a.W;
  auto slot_of = [&](int i) { return reinterpret_cast<float*>(sm + C::OFF_R + (uint32_t)(q * C::NS + i % C::NS) * C::CHUNK); };
  auto chunk_rows = [&](int i) { return max(0, min(8, T.rcnt - (r0 + 8 * (i & 3)))); };
  auto issue_item = [&](int i) {
    if (i < n_items) {
      const int w = i >> 2, nv = chunk_rows(i);
      const int64_t o = (int64_t)(T.row0 + r0 + 8 * (i & 3)) * L.ld + L.off + (int64_t)T.seg * kMCols;
      const float* gp = a.G[w] + o;
      const float* bp = a.B + (int64_t)w * a.total + o;
      float* dst = slot_of(i);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = jq + 128 * h;  // float4 e of the chunk: row e / 32, columns 4 (e % 32) ..
        const int k = e >> 5, c4 = 4 * (e & 31);
        if (k < nv && c4 < segcols) {
          cp_async_16(dst + 128 * k + c4, gp + (int64_t)k * L.ld + c4);
          cp_async_16(dst + 1024 + 128 * k + c4, bp + (int64_t)k * L.ld + c4);
        }
      }
    }
    cp_async_commit();  // one group per item (empty past the last one)
  };
#pragma unroll
  for (int i = 0; i < C::NS - 1; ++i) issue_item(i);
  for (int w = 0; w < a.W; ++w) {
    if (prev && w + 1 < a.W) stage_qw(w + 1);  // its buffer's last reader, worker w - 1's MMA, is done
    fence_async_smem();
    tc_fence_before();
    __syncthreads();  // staged; and every thread is done with D of worker w - 1
    tc_fence_after();
    if (prev && w + 1 < a.W && tid == 0) issue_e(w + 1);
    if (prev && !mbar_wait(&s_mbar[w & 1], (uint32_t)((w >> 1) & 1))) {
      ok = false;
      if (lane == 0 && a.sync) atomicCAS(a.sync + 2, 0u, 2u);
    }
    tc_fence_after();
    if (!__syncthreads_and(ok ? 1 : 0)) {  // a wait ran out: abandon the tile
      ok = false;                          // (in every thread)
      break;
    }
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      const int i = 4 * w + ch;
      float d[8];
      if (prev)
        tmem_ld8(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(w & 1) * kMRows + (uint32_t)(r0 + 8 * ch), d);
      // this thread's copies of item i have landed; after the barrier every
      // thread's have, and every thread is done with item i - 1's slot
      cp_async_wait<C::NS - 2>();
      named_barrier(1 + q, 128);
      issue_item(i + C::NS - 1);  // into item i - 1's slot
      const int rfirst = r0 + 8 * ch;
      const int nv = col_in ? chunk_rows(i) : 0;
      const float* sg = slot_of(i) + cl;
      float* bp = a.B + (int64_t)w * a.total + (int64_t)(T.row0 + rfirst) * L.ld + L.off + col;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float g = k < nv ? sg[128 * k] : 0.f;
        const float b = k < nv ? sg[1024 + 128 * k] : 0.f;
        float m = prev ? g + (b - d[k]) : g + b;
        if (col >= L.m) m = 0.f;  // the row padding stays zero
        if (k < nv) *bp = m;
        bp += L.ld;
        msum[8 * ch + k] += m;
      }
    }
  }
  cp_async_wait<0>();  // no copy is in flight when the space is reused or the CTA leaves
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!ok) {
    if (warp == 0) tmem_free(tmem, C::TMEM_COLS);
    return;
  }
  // P_tile = Msum Q: Msum (hi, lo) as the A operand (K = the 128 columns,
  // over the Q_w' buffers) and Q^T (hi, lo) as the B operand
  {
    unsigned char* mhi = sm + C::OFF_U;
    unsigned char* mlo = mhi + C::MS_P;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float h, l;
      tf32_split(msum[i], h, l);
      const int r = r0 + i;
      const uint32_t o = (uint32_t)(r >> 3) * C::M_SBO + (uint32_t)(cl >> 2) * C::M_LBO + (uint32_t)(r & 7) * 16 +
                         (uint32_t)(cl & 3) * 4;
      *reinterpret_cast<float*>(mhi + o) = h;
      *reinterpret_cast<float*>(mlo + o) = l;
    }
    const float* q = a.Qbar + L.q_off + (int64_t)T.seg * kMCols * RP;
    constexpr int K4 = RP / 4;
    for (int e = tid; e < kMCols * K4; e += blockDim.x) {
      const int c = e / K4, k4 = e - c * K4;
      const float4 v = c < segcols ? __ldg(reinterpret_cast<const float4*>(q + (int64_t)c * RP) + k4) : zero4();
      const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float h, l;
        tf32_split(x[i], h, l);
        const uint32_t o = umma_off(4 * k4 + i, c, kMCols);
        *reinterpret_cast<float*>(sm + C::OFF_Q + o) = h;
        *reinterpret_cast<float*>(sm + C::OFF_Q + C::OP + o) = l;
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    constexpr uint32_t id = umma_idesc_tf32(kMRows, RP);
    const uint32_t d = tmem + 2u * kMRows;
    const uint32_t ahi = base + C::OFF_U, alo = ahi + C::MS_P;
    const uint32_t bhi = base + C::OFF_Q, blo = bhi + C::OP;
#pragma unroll 1
    for (int ks = 0; ks < kMCols / 8; ++ks) {
      const uint32_t oa = (uint32_t)ks * 2 * C::M_LBO, ob = (uint32_t)ks * 256;
      umma_tf32(d, umma_sdesc_los(ahi + oa, C::M_LBO, C::M_SBO), umma_sdesc(bhi + ob, kMCols), id, ks > 0 ? 1u : 0u);
      umma_tf32(d, umma_sdesc_los(ahi + oa, C::M_LBO, C::M_SBO), umma_sdesc(blo + ob, kMCols), id, 1u);
      umma_tf32(d, umma_sdesc_los(alo + oa, C::M_LBO, C::M_SBO), umma_sdesc(bhi + ob, kMCols), id, 1u);
    }
    umma_commit(&s_mbar[2]);
  }
  float* s_prow = reinterpret_cast<float*>(sm + C::OFF_P);  // the Phat' tile is no longer read
  double* s_gram = reinterpret_cast<double*>(sm + C::OFF_P + (uint32_t)kMRows * RP * 4);
  if (!mbar_wait(&s_mbar[2], 0u)) {
    ok = false;
    if (tid == 0 && a.sync) atomicCAS(a.sync + 2, 0u, 2u);
  }
  tc_fence_after();
  if (ok && warp < 4) {  // P rows: TMEM lane = row here
    const int r = 32 * warp + lane;
#pragma unroll
    for (int h = 0; h < RP / 16; ++h) {
      float p[16];
      tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + 2u * kMRows + 16u * h, p);
      if (r < T.rcnt)
#pragma unroll
        for (int k = 0; k < 16; ++k) s_prow[r * RP + 16 * h + k] = p[k];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tmem, C::TMEM_COLS);
  if (!__syncthreads_and(ok ? 1 : 0)) return;
  p1_rows_done<RP>(a, L, T, s_prow, s_gram, &s_flag, nullptr);
}

// ----------------------------------------------------------------------------
// back-project on the tensor cores (r >= 16)
// ----------------------------------------------------------------------------
//
// Q_w (partial over a row tile) = M_w^T Phat: per 128-row chunk and worker,
// D_w (128 columns x r, TMEM; lane = column) += M_w[chunk]^T Phat[chunk] in
// error-compensated TF32, D_w accumulating over the tile's chunks in TMEM
// columns w r.  The A operand (M_w^T: the segment's 128 columns x 128 rows,
// K-major) is written by the CUDA cores, transposed: a warp loads 4 rows x
// 32 columns (float4 per lane, 128-byte rows) and stores each value's hi and
// lo parts; its 8-column core-matrix groups are BSBO bytes apart, 16 more
// than packed, so that those scattered 4-byte stores hit 32 distinct banks.
// The B operand is the chunk's Phat rows (r x 128, K-major).  Each thread
// loads its 8 float4 of the next (chunk, worker) while the tensor cores run
// the current one.  At the end every worker's D is read from TMEM as the
// tile's partial Q_w; the row tiles' partials are summed as in the CUDA-core
// back-project (last arriver per segment and worker, then Qbar).
constexpr int kBThreads = 512;    // 16 warps
constexpr int kBRows = 128;       // rows of a chunk: the K of one round of MMAs

template <int RP>
struct BmmaCfg {
  static_assert(RP == 16 || RP == 32, "tensor-core back-project tiles are for padded ranks 16 and 32");
  static constexpr uint32_t SBO = (kBRows / 4) * 128 + 16;       // A: 8-column groups apart (padded)
  static constexpr uint32_t A_BYTES = (kMCols / 8) * SBO;        // one copy (hi or lo) of A
  static constexpr uint32_t B_SBO = (kBRows / 4) * 128;          // B: 8-rank groups apart
  static constexpr uint32_t B_BYTES = (uint32_t)(RP / 8) * B_SBO;  // one copy of B (r x 128)
  static constexpr uint32_t OFF_A = 0;                             // A hi, then lo
  static constexpr uint32_t OFF_B = 2 * A_BYTES;                   // B hi, then lo
  static constexpr uint32_t SMEM = OFF_B + 2 * B_BYTES;
  static_assert(SMEM <= 227 * 1024, "fits the shared memory of one CTA");
  static_assert(A_BYTES % 16 == 0 && B_BYTES % 16 == 0, "operands start on 16-byte boundaries");
};

// Byte offset of element (m, k) of the padded K-major A operand (K = 128).
template <int RP>
__device__ __forceinline__ uint32_t bmma_a_off(int m, int k) {
  return (uint32_t)(m >> 3) * BmmaCfg<RP>::SBO + (uint32_t)(k >> 2) * 128 + (uint32_t)(m & 7) * 16 + (uint32_t)(k & 3) * 4;
}

template <int RP>
__global__ void __launch_bounds__(kBThreads, 1) p3m_kernel(const StepArgs a) {
  using C = BmmaCfg<RP>;
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t s_mbar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_flag;
  pdl_enter();
  const Tile t = a.tiles[blockIdx.x];
  const LayerDev L = a.layers[t.layer];  // by value: stores cannot alias it
  const int rt = t.a, seg = t.b;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = rt * L.r3;
  const int nrows = min(L.r3, L.n - row0);
  const int nchunks = (nrows + kBRows - 1) / kBRows;
  const int segcols = min(kMCols, L.ld - seg * kMCols);
  const uint32_t base = smem_u32(sm);
  if (warp == 0) tmem_alloc(&s_tmem, kBmmaTmemCols);
  if (tid == 0) mbar_init(&s_mbar);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // this thread's 8 float4 of a chunk: rows 8 warp + 4 (u & 1) + lane / 8,
  // float4 column 8 (u / 2) + lane % 8, u = 0..7
  const int n_it = nchunks * a.W;  // iteration it = chunk it / W, worker it % W
  float4 v[8];
  auto load_it = [&](int it) {
    const int c = it / a.W, w = it - c * a.W;
    const float* bw = a.B + (int64_t)w * a.total + L.off + (int64_t)seg * kMCols;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = 8 * warp + 4 * (u & 1) + (lane >> 3);
      const int c4 = 4 * (8 * (u >> 1) + (lane & 7));
      const int row = c * kBRows + r;
      v[u] = (row < nrows && c4 < segcols)
                 ? __ldcs(reinterpret_cast<const float4*>(bw + (int64_t)(row0 + row) * L.ld + c4))
                 : zero4();
    }
  };
  auto store_a = [&]() {
    unsigned char* ahi = sm + C::OFF_A;
    unsigned char* alo = ahi + C::A_BYTES;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = 8 * warp + 4 * (u & 1) + (lane >> 3);
      const int m0 = 4 * (8 * (u >> 1) + (lane & 7));
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float h, l;
        tf32_split(x[j], h, l);
        const uint32_t o = bmma_a_off<RP>(m0 + j, r);
        *reinterpret_cast<float*>(ahi + o) = h;
        *reinterpret_cast<float*>(alo + o) = l;
      }
    }
  };
  // the chunk's Phat rows as the B operand (rank n, row k), hi and lo
  auto stage_b = [&](int c) {
    constexpr int K4 = RP / 4;
    const float* ph = a.Phat + L.p_off + (int64_t)(row0 + c * kBRows) * RP;
    const int rows = min(kBRows, nrows - c * kBRows);
    for (int e = tid; e < kBRows * K4; e += kBThreads) {
      const int k = e / K4, n4 = e - k * K4;
      const float4 p = k < rows ? __ldg(reinterpret_cast<const float4*>(ph + (int64_t)k * RP) + n4) : zero4();
      const float x[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float h, l;
        tf32_split(x[j], h, l);
        const int n = 4 * n4 + j;
        const uint32_t o = (uint32_t)(n >> 3) * C::B_SBO + (uint32_t)(k >> 2) * 128 + (uint32_t)(n & 7) * 16 + (uint32_t)(k & 3) * 4;
        *reinterpret_cast<float*>(sm + C::OFF_B + o) = h;
        *reinterpret_cast<float*>(sm + C::OFF_B + C::B_BYTES + o) = l;
      }
    }
  };

  bool ok = true;
  if (n_it > 0) load_it(0);
  for (int it = 0; it < n_it; ++it) {
    const int c = it / a.W, w = it - c * a.W;
    // the tensor cores are done with the operands of iteration it - 1
    if (it > 0 && !mbar_wait(&s_mbar, (uint32_t)((it - 1) & 1))) {
      ok = false;
      if (lane == 0 && a.sync) atomicCAS(a.sync + 2, 0u, 2u);
    }
    tc_fence_after();
    if (!__syncthreads_and(ok ? 1 : 0)) {
      ok = false;
      break;
    }
    if (w == 0) stage_b(c);
    store_a();
    if (it + 1 < n_it) load_it(it + 1);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      constexpr uint32_t id = umma_idesc_tf32(kMCols, RP);
      const uint32_t d = tmem + (uint32_t)(w * RP);
      const uint32_t ahi = base + C::OFF_A, alo = ahi + C::A_BYTES;
      const uint32_t bhi = base + C::OFF_B, blo = bhi + C::B_BYTES;
#pragma unroll 1
      for (int ks = 0; ks < kBRows / 8; ++ks) {
        const uint32_t o = (uint32_t)ks * 256;
        const uint32_t acc = (c > 0 || ks > 0) ? 1u : 0u;
        umma_tf32(d, umma_sdesc_los(ahi + o, 128, C::SBO), umma_sdesc_los(bhi + o, 128, C::B_SBO), id, acc);
        umma_tf32(d, umma_sdesc_los(ahi + o, 128, C::SBO), umma_sdesc_los(blo + o, 128, C::B_SBO), id, 1u);
        umma_tf32(d, umma_sdesc_los(alo + o, 128, C::SBO), umma_sdesc_los(bhi + o, 128, C::B_SBO), id, 1u);
      }
      umma_commit(&s_mbar);
    }
  }
  if (ok && n_it > 0 && !mbar_wait(&s_mbar, (uint32_t)((n_it - 1) & 1))) {
    ok = false;
    if (tid == 0 && a.sync) atomicCAS(a.sync + 2, 0u, 2u);
  }
  tc_fence_after();
  // every worker's D: the tile's partial Q_w (TMEM lane = column)
  if (ok) {
    const int g = warp & 3, cl = 32 * g + lane;
    for (int w = warp >> 2; w < a.W; w += 4) {
      float q[RP];
      if constexpr (RP == 32) {
        tmem_ld32(tmem + ((uint32_t)(32 * g) << 16) + (uint32_t)(w * RP), q);
      } else {
        tmem_ld16(tmem + ((uint32_t)(32 * g) << 16) + (uint32_t)(w * RP), q);
      }
      if (cl < segcols) {
        float4* dst = reinterpret_cast<float4*>(a.qpart + L.qpart_off +
                                                ((int64_t)(rt * a.W + w) * L.ld + seg * kMCols + cl) * RP);
#pragma unroll
        for (int k4 = 0; k4 < RP / 4; ++k4) dst[k4] = make_float4(q[4 * k4], q[4 * k4 + 1], q[4 * k4 + 2], q[4 * k4 + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tmem, kBmmaTmemCols);
  if (!__syncthreads_and(ok ? 1 : 0)) return;
  for (int w = 0; w < a.W; ++w)
    if (cta_arrive_last(a.counters + L.cnt_off + L.c_p3 + seg * a.W + w, (unsigned)L.t3r, &s_flag))
      qf_segment_worker<RP>(a, L, seg, w, &s_flag, nullptr);
}

}  // namespace psgd
