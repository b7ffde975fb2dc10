// The project phase for padded ranks 16 and 32 on the tensor cores (tcgen05).
//
// At r >= 16 the project tile's arithmetic outgrows its bytes: per element
// and worker, the error rebuild E = B - Phat' Q_w'^T is r multiply-adds, and
// the CUDA-core kernel is bound by feeding those from shared memory.  Here
// the rebuild is a tensor-core product per (tile, worker):
//
//   D_w (128 x 128, TMEM) = Phat'_tile (128 x r) Q_w'_segment^T (r x 128)
//
// in error-compensated TF32 (hi/lo split, three MMAs per K step: float32
// accuracy), and the tile's share of P is one more product after the
// workers, P_tile (128 x r) = Msum (128 x 128) Q_segment (128 x r), with
// Msum = sum_w M_w (P is linear in M).  The threads stream G and B with
// coalesced float4 loads, take D_w from TMEM (through a shared-memory
// exchange, so that each thread gets the columns it loaded), form
// M_w = G_w + B_w - D_w, store it to B_w and add it to Msum.
//
// A CTA owns 128 rows (the 128 TMEM lanes) x one segment (128 columns) and
// loops over the workers; worker w + 1's Q_w' rows are staged and its MMAs
// issued while worker w's rows are combined (D in two TMEM buffers).  Every
// wait on the tensor cores is bounded; one that runs out marks the step's
// status word (the host reports it) and the tile is abandoned.
#pragma once

#include "psgd_kernels.cuh"
#include "psgd_umma.cuh"

namespace psgd {

constexpr int kMThreads = 512;     // 16 warps: 4 TMEM lane groups x 4 column quarters
constexpr int kMRows = 128;        // rows of a tile (the TMEM lanes)
constexpr int kMCols = kSeg * 4;   // columns of a tile (one segment)
constexpr int kXRow = kMCols + 4;  // exchange row stride in floats (conflict-free float4 reads)

template <int RP>
struct MmaCfg {
  static_assert(RP == 16 || RP == 32, "tensor-core project tiles are for padded ranks 16 and 32");
  static constexpr uint32_t A1 = (uint32_t)kMRows * RP * 4;  // one copy (hi or lo) of the Phat' tile
  static constexpr uint32_t QB = (uint32_t)kMCols * RP * 4;  // one copy of Q_w' (128 x r) or of Q^T (r x 128)
  static constexpr uint32_t QW = 2 * QB;                      // a Q_w' buffer: hi, lo
  static constexpr uint32_t XB = (uint32_t)kMRows * kXRow * 4;
  static constexpr uint32_t MS = (uint32_t)kMRows * kMCols * 4;  // one copy of Msum
  static constexpr uint32_t OFF_A1 = 0;           // Phat' hi, lo; later the P rows and the Gram scratch
  static constexpr uint32_t OFF_Q = 2 * A1;       // Q^T hi, lo
  static constexpr uint32_t OFF_U = OFF_Q + 2 * QB;  // { Q_w' buffers 0, 1; exchange } or { Msum hi, lo }
  static constexpr uint32_t OFF_X = OFF_U + 2 * QW;
  static constexpr uint32_t U_BYTES = (2 * QW + XB > 2 * MS) ? 2 * QW + XB : 2 * MS;
  static constexpr uint32_t SMEM = OFF_U + U_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;  // D of two workers (2 x 128) and the P tile (r)
  static_assert((uint32_t)kMRows * RP * 4 + RP * RP * 8 <= 2 * A1, "P rows and Gram scratch fit over the Phat' tile");
};

// Stages a rows x RP row-major float32 block (rows past `valid` as zeros) as
// the hi and lo copies of a K-major operand with K = RP.
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
  const int c4 = T.seg * kSeg + lane;  // this thread's float4 column; its rows are warp + 16 j
  const bool col_ok = c4 < L.F;
  const int segcols = min(kMCols, L.ld - T.seg * kMCols);
  const bool prev = T.prev;
  const uint32_t base = smem_u32(sm);

  if (warp == 0) tmem_alloc(&s_tmem, C::TMEM_COLS);
  if (tid == 0) {
    mbar_init(&s_mbar[0]);
    mbar_init(&s_mbar[1]);
    mbar_init(&s_mbar[2]);
  }
  // the operands every worker shares: the previous Phat rows of the tile and
  // Q^T of the segment; and worker 0's Q_w'
  stage_kmajor_rows<RP>(sm + C::OFF_A1, sm + C::OFF_A1 + C::A1, a.Phat + L.p_off + (int64_t)T.row0 * RP, kMRows,
                        T.rcnt, !prev);
  {
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
        *reinterpret_cast<float*>(sm + C::OFF_Q + C::QB + o) = l;
      }
    }
  }
  auto stage_qw = [&](int w) {
    unsigned char* buf = sm + C::OFF_U + (w & 1) * C::QW;
    stage_kmajor_rows<RP>(buf, buf + C::QB, a.Qw + (int64_t)w * a.q_total + L.q_off + (int64_t)T.seg * kMCols * RP,
                          kMCols, segcols, false);
  };
  if (prev) stage_qw(0);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  // D_w = Phat'_tile Q_w'^T into TMEM columns (w & 1) * 128, hi hi + hi lo + lo hi
  auto issue_e = [&](int w) {
    constexpr uint32_t id = umma_idesc_tf32(kMRows, kMCols);
    const uint32_t d = tmem + (uint32_t)(w & 1) * kMCols;
    const uint32_t ahi = base + C::OFF_A1, alo = ahi + C::A1;
    const uint32_t bhi = base + C::OFF_U + (uint32_t)(w & 1) * C::QW, blo = bhi + C::QB;
#pragma unroll
    for (int ks = 0; ks < RP / 8; ++ks) {
      const uint32_t o = (uint32_t)ks * 256;
      umma_tf32(d, umma_sdesc(ahi + o, RP), umma_sdesc(bhi + o, RP), id, ks > 0 ? 1u : 0u);
      umma_tf32(d, umma_sdesc(ahi + o, RP), umma_sdesc(blo + o, RP), id, 1u);
      umma_tf32(d, umma_sdesc(alo + o, RP), umma_sdesc(bhi + o, RP), id, 1u);
    }
    umma_commit(&s_mbar[w & 1]);
  };
  if (prev && tid == 0) issue_e(0);

  float msum[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) msum[j][0] = msum[j][1] = msum[j][2] = msum[j][3] = 0.f;
  float* s_x = reinterpret_cast<float*>(sm + C::OFF_X);
  for (int w = 0; w < a.W; ++w) {
    // this worker's G and B rows first: their loads fly while the MMA runs
    const float* Gw = a.G[w] + L.off + 4 * c4;
    float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * c4;
    float4 g[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = warp + 16 * j;
      g[j] = b[j] = zero4();
      if (col_ok && r < T.rcnt) {
        const int64_t o = (int64_t)(T.row0 + r) * L.ld;
        g[j] = __ldcs(reinterpret_cast<const float4*>(Gw + o));
        b[j] = __ldcs(reinterpret_cast<const float4*>(Bw + o));
      }
    }
    if (prev && w + 1 < a.W) stage_qw(w + 1);  // its buffer's last reader, worker w - 1's MMA, is done
    if (prev) {
      if (!mbar_wait(&s_mbar[w & 1], (uint32_t)((w >> 1) & 1))) {
        ok = false;
        if (lane == 0 && a.sync) atomicCAS(a.sync + 2, 0u, 2u);
      }
      tc_fence_after();
      // D_w: warp (lane group warp % 4, column quarter warp / 4) -> exchange rows
      if (ok) {
        const uint32_t src = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(w & 1) * kMCols + 32u * (warp >> 2);
        float4* dst = reinterpret_cast<float4*>(s_x + (32 * (warp & 3) + lane) * kXRow + 32 * (warp >> 2));
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two halves of 16 columns: fewer live registers
          float d[16];
          tmem_ld16(src + 16u * h, d);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[4 * h + i] = make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!__syncthreads_and(ok ? 1 : 0)) {  // a tensor-core wait ran out: abandon the tile
      ok = false;                          // (in every thread)
      break;
    }
    if (prev && w + 1 < a.W && tid == 0) issue_e(w + 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = warp + 16 * j;
      float4 m = make_float4(g[j].x + b[j].x, g[j].y + b[j].y, g[j].z + b[j].z, g[j].w + b[j].w);
      if (prev) {
        const float4 dv = reinterpret_cast<const float4*>(s_x + r * kXRow)[lane];
        m = make_float4(g[j].x + (b[j].x - dv.x), g[j].y + (b[j].y - dv.y), g[j].z + (b[j].z - dv.z),
                        g[j].w + (b[j].w - dv.w));
      }
      const int col = 4 * c4;  // the row padding stays zero
      if (col >= L.m) m.x = 0.f;
      if (col + 1 >= L.m) m.y = 0.f;
      if (col + 2 >= L.m) m.z = 0.f;
      if (col + 3 >= L.m) m.w = 0.f;
      if (col_ok && r < T.rcnt) reinterpret_cast<float4*>(Bw + (int64_t)(T.row0 + r) * L.ld)[0] = m;
      msum[j][0] += m.x;
      msum[j][1] += m.y;
      msum[j][2] += m.z;
      msum[j][3] += m.w;
    }
    __syncthreads();  // the exchange is free for the next worker
  }
  if (!ok) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tmem, C::TMEM_COLS);
    return;
  }
  // P_tile = Msum Q: Msum (hi, lo) as the A operand, K = the 128 columns
  {
    unsigned char* mhi = sm + C::OFF_U;
    unsigned char* mlo = mhi + C::MS;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float4 h, l;
      tf32_split(msum[j][0], h.x, l.x);
      tf32_split(msum[j][1], h.y, l.y);
      tf32_split(msum[j][2], h.z, l.z);
      tf32_split(msum[j][3], h.w, l.w);
      const uint32_t o = umma_off(warp + 16 * j, 4 * lane, kMCols);
      *reinterpret_cast<float4*>(mhi + o) = h;
      *reinterpret_cast<float4*>(mlo + o) = l;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    constexpr uint32_t id = umma_idesc_tf32(kMRows, RP);
    const uint32_t d = tmem + 2u * kMCols;
    const uint32_t ahi = base + C::OFF_U, alo = ahi + C::MS;
    const uint32_t bhi = base + C::OFF_Q, blo = bhi + C::QB;
#pragma unroll 4
    for (int ks = 0; ks < kMCols / 8; ++ks) {
      const uint32_t o = (uint32_t)ks * 256;
      umma_tf32(d, umma_sdesc(ahi + o, kMCols), umma_sdesc(bhi + o, kMCols), id, ks > 0 ? 1u : 0u);
      umma_tf32(d, umma_sdesc(ahi + o, kMCols), umma_sdesc(blo + o, kMCols), id, 1u);
      umma_tf32(d, umma_sdesc(alo + o, kMCols), umma_sdesc(bhi + o, kMCols), id, 1u);
    }
    umma_commit(&s_mbar[2]);
  }
  float* s_prow = reinterpret_cast<float*>(sm + C::OFF_A1);  // the Phat' tile is no longer read
  double* s_gram = reinterpret_cast<double*>(sm + C::OFF_A1 + (uint32_t)kMRows * RP * 4);
  if (!mbar_wait(&s_mbar[2], 0u)) {
    ok = false;
    if (tid == 0 && a.sync) atomicCAS(a.sync + 2, 0u, 2u);
  }
  tc_fence_after();
  if (ok && warp < 4) {
    float p[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 2u * kMCols, p);
    const int r = 32 * warp + lane;
    if (r < T.rcnt)
#pragma unroll
      for (int k = 0; k < RP; ++k) s_prow[r * RP + k] = p[k];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tmem, C::TMEM_COLS);
  if (!__syncthreads_and(ok ? 1 : 0)) return;
  p1_rows_done<RP>(a, L, T, s_prow, s_gram, &s_flag, nullptr);
}

}  // namespace psgd
