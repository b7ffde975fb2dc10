// The one-pass project phase (padded rank <= 4) on thread-block clusters.
//
// PowerSGD's back-projection Q_w = M_w^T Phat with Phat = P R^-1 (one
// Cholesky-QR pass) equals (M_w^T P) R^-1.  Row i of P = sum_w M_w Q needs
// only row i of every worker's M, so once a row block's P rows are complete,
// Y_w += M_w[rows]^T P[rows] can be accumulated while those M rows are still
// on chip -- and the back-project phase no longer reads M from HBM: it forms
// Q_w = Y_w R^-1 from the (small) Y partials.  The one condition is P's
// conditioning (the rounding of Y is amplified by about kappa(P)); the
// factor's last arriver checks kappa_F(R) and otherwise leaves the layer to
// the two-pass back-project.
//
// A layer's row is split over cw CTAs (column slices of yfc float4 columns,
// all W workers each); cw is a power of two dividing the cluster size, and a
// cluster of kYClusterMax CTAs holds kYClusterMax / cw such subgroups, each
// on its own row group of ryg rows.  Per block of R rows a CTA
//   1. streams G and B of its slice (128-bit loads), rebuilds E = B - Phat'
//      Q_w'^T, stores M = G + E to B, and sums its share of the block's P rows
//      (warp butterfly, then a fixed-order sum over the warps);
//   2. pushes that share into every subgroup member's shared memory
//      (st.shared::cluster) and arrives on the cluster barrier (release);
//   3. streams the next block (step 1) while the barrier completes;
//   4. waits (acquire), sums the members' shares in rank order -- every member
//      gets the same P rows, bit for bit -- and re-reads its own M rows of the
//      block (just written: an L2 hit) to accumulate Y in shared memory.
// The subgroup's first CTA stores the P rows and keeps the block's float64
// Gram sums.  At the end of the row group every CTA stores its slice of the
// group's Y partial, and the first CTA runs the Gram tail (gram_finish) over
// the layer's row groups.
#pragma once

#include "psgd_kernels.cuh"

namespace psgd {

template <int RP>
struct YCfg {
  static constexpr int R = y_rows(RP);         // rows of a block
  static constexpr int PT = y_pairs_max(RP);   // (float4 column, worker) pairs per thread at most
  static constexpr int RU = R < 4 ? R : 4;     // rows whose G and B loads are in flight together
  static constexpr int NV = R * RP;            // P values of a block
  static constexpr int NW = kYThreads / 32;
  // dynamic shared memory: the Y accumulators, PT x RP float4 per thread
  static constexpr size_t SMEM = (size_t)PT * RP * kYThreads * sizeof(float4);
  static_assert(NV == 16, "a block's P values are one 16-value warp butterfly");
};

__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned cluster_index() {
  unsigned r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Cluster barrier, split: arrive (release: this thread's earlier writes,
// shared::cluster ones included, are visible to the cluster once every
// thread has arrived) and wait (acquire).  Every thread of every CTA of the
// cluster executes both, the same number of times.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Stores v at the shared-memory location of `local` in the CTA of cluster rank `rank`.
__device__ __forceinline__ void st_cluster_f32(const float* local, unsigned rank, float v) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(r), "f"(v) : "memory");
}

// The geometry of one CTA of the one-pass project.
struct YTile {
  int sub, kl;              // subgroup of the cluster, rank within the subgroup
  int g;                    // row group (>= nyg: an idle subgroup)
  int row_begin, row_end;   // rows of the group (empty when idle)
  int nblk;                 // blocks of R rows per group (the same in the whole cluster)
  int f0, nf, ps;           // first float4 column, float4 columns and pairs of the slice
};

// Step 1 for block b: E, M (stored to B) and this thread's share of the
// block's P values, pp[u * RP + k] (row u of the block, rank k).
template <int RP>
__device__ __forceinline__ void y_phase1(const StepArgs& a, const LayerDev& L, const YTile& Y, int b,
                                         float (&pp)[YCfg<RP>::NV]) {
  using C = YCfg<RP>;
  constexpr int R = C::R, RU = C::RU;
#pragma unroll
  for (int i = 0; i < C::NV; ++i) pp[i] = 0.f;
  const int r0 = Y.row_begin + b * R;
  const bool prev = a.has_prev != 0;
  const float* Pprev = a.Phat + L.p_off + (int64_t)r0 * RP;
  for (int j = 0; j < C::PT; ++j) {
    const int p = (int)threadIdx.x + j * kYThreads;
    if (p >= Y.ps) break;
    const int w = p / Y.nf, f = Y.f0 + p % Y.nf;
    const float* Gw = a.G[w] + L.off + 4 * f;
    float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * f;
    // this pair's 4 rows of Q and of Q_w' (rows 4f .. 4f + 3 of ld x RP)
    float qv[4][RP], qw[4][RP];
    {
      const float4* sq = reinterpret_cast<const float4*>(a.Qbar + L.q_off + (int64_t)(4 * f) * RP);
      const float4* sw = reinterpret_cast<const float4*>(a.Qw + (int64_t)w * a.q_total + L.q_off + (int64_t)(4 * f) * RP);
      float* fq = &qv[0][0];
      float* fw = &qw[0][0];
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const float4 v = __ldg(sq + i);
        fq[4 * i] = v.x;
        fq[4 * i + 1] = v.y;
        fq[4 * i + 2] = v.z;
        fq[4 * i + 3] = v.w;
        const float4 x = prev ? __ldg(sw + i) : zero4();
        fw[4 * i] = x.x;
        fw[4 * i + 1] = x.y;
        fw[4 * i + 2] = x.z;
        fw[4 * i + 3] = x.w;
      }
    }
    const bool tailc = (f == L.F - 1) && (L.tail < 4);
#pragma unroll
    for (int u0 = 0; u0 < R; u0 += RU) {
      float4 gv[RU], bv[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int row = r0 + u0 + u;
        if (row < Y.row_end) {
          gv[u] = __ldcs(reinterpret_cast<const float4*>(Gw + (int64_t)row * L.ld));
          bv[u] = __ldcs(reinterpret_cast<const float4*>(Bw + (int64_t)row * L.ld));
        } else {
          gv[u] = zero4();
          bv[u] = zero4();
        }
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int row = r0 + u0 + u;
        if (row < Y.row_end) {
          // E = B - Phat' Q_w'^T, k ascending (the chain of the error read-back)
          float e0 = bv[u].x, e1 = bv[u].y, e2 = bv[u].z, e3 = bv[u].w;
          if (prev) {
#pragma unroll
            for (int k = 0; k < RP; ++k) {
              const float ph = __ldg(Pprev + (u0 + u) * RP + k);
              e0 = fmaf(-ph, qw[0][k], e0);
              e1 = fmaf(-ph, qw[1][k], e1);
              e2 = fmaf(-ph, qw[2][k], e2);
              e3 = fmaf(-ph, qw[3][k], e3);
            }
          }
          float m0 = gv[u].x + e0, m1 = gv[u].y + e1, m2 = gv[u].z + e2, m3 = gv[u].w + e3;
          if (tailc) {
            if (L.tail < 2) m1 = 0.f;
            if (L.tail < 3) m2 = 0.f;
            m3 = 0.f;
          }
          // a plain store: the line stays in L2 for step 4's read
          *reinterpret_cast<float4*>(Bw + (int64_t)row * L.ld) = make_float4(m0, m1, m2, m3);
#pragma unroll
          for (int k = 0; k < RP; ++k) {
            float t = m0 * qv[0][k];
            t = fmaf(m1, qv[1][k], t);
            t = fmaf(m2, qv[2][k], t);
            t = fmaf(m3, qv[3][k], t);
            pp[(u0 + u) * RP + k] += t;
          }
        }
      }
    }
  }
}

// The CTA's share of the block's P values: warp butterfly, then (after the
// caller's barrier) the fixed-order sum over the warps.  s_red_b: NW x NV.
template <int RP>
__device__ __forceinline__ void y_reduce_warps(float (&pp)[YCfg<RP>::NV], float* s_red_b) {
  using C = YCfg<RP>;
  float tot;
  const int jv = warp_reduce_multi<C::NV>(pp, tot);
  if ((threadIdx.x & 1) == 0) s_red_b[(threadIdx.x >> 5) * C::NV + jv] = tot;
}

// Thread v < NV: the CTA's share of P value v, pushed into slot kl of every
// member of the subgroup (ranks sub * cw .. + cw - 1).
template <int RP>
__device__ __forceinline__ void y_push(const YTile& Y, int cw, const float* s_red_b, float* s_slot_b) {
  using C = YCfg<RP>;
  const int v = threadIdx.x;
  float s = 0.f;
#pragma unroll
  for (int wv = 0; wv < C::NW; ++wv) s += s_red_b[wv * C::NV + v];
  float* dst = s_slot_b + Y.kl * C::NV + v;
  for (int t = 0; t < cw; ++t) st_cluster_f32(dst, (unsigned)(Y.sub * cw + t), s);
}

// Step 4 for block b: Y += M[rows]^T P[rows] over this thread's pairs.
// s_p: the block's P values (R x RP); s_y: PT x RP x kYThreads float4.
template <int RP>
__device__ __forceinline__ void y_phase2(const StepArgs& a, const LayerDev& L, const YTile& Y, int b,
                                         const float* s_p, float4* s_y) {
  using C = YCfg<RP>;
  constexpr int R = C::R;
  const int r0 = Y.row_begin + b * R;
  for (int j = 0; j < C::PT; ++j) {
    const int p = (int)threadIdx.x + j * kYThreads;
    if (p >= Y.ps) break;
    const int w = p / Y.nf, f = Y.f0 + p % Y.nf;
    const float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * f;
    float4 m[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int row = r0 + u;
      // this thread stored these M values in step 1 (program order)
      m[u] = row < Y.row_end ? __ldcg(reinterpret_cast<const float4*>(Bw + (int64_t)row * L.ld)) : zero4();
    }
    float4 y[RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) y[k] = s_y[(j * RP + k) * kYThreads + threadIdx.x];
#pragma unroll
    for (int u = 0; u < R; ++u) {
#pragma unroll
      for (int k = 0; k < RP; ++k) {
        const float pv = s_p[u * RP + k];
        y[k].x = fmaf(m[u].x, pv, y[k].x);
        y[k].y = fmaf(m[u].y, pv, y[k].y);
        y[k].z = fmaf(m[u].z, pv, y[k].z);
        y[k].w = fmaf(m[u].w, pv, y[k].w);
      }
    }
#pragma unroll
    for (int k = 0; k < RP; ++k) s_y[(j * RP + k) * kYThreads + threadIdx.x] = y[k];
  }
}

template <int RP>
__global__ void __launch_bounds__(kYThreads, 2) p1c_kernel(const StepArgs a) {
  using C = YCfg<RP>;
  constexpr int R = C::R, NV = C::NV, NG = Cfg<RP>::NG;
  extern __shared__ float4 s_y[];                   // the Y accumulators
  __shared__ float s_slot[2][kYClusterMax * NV];    // the subgroup's shares of a block's P values
  __shared__ float s_red[2][C::NW * NV];            // the warps' shares
  __shared__ float s_prow[2][NV];                   // a block's P values
  __shared__ double s_gram[RP * RP];
  __shared__ int s_flag;
  pdl_enter();
  const Tile t = a.tiles[cluster_index()];
  const LayerDev L = a.layers[t.layer];  // by value: stores to B cannot alias it
  const int cw = L.cw;
  const unsigned rank = cluster_ctarank();
  YTile Y;
  Y.sub = (int)rank / cw;
  Y.kl = (int)rank % cw;
  Y.g = t.a + Y.sub;
  Y.row_begin = Y.g * L.ryg;
  Y.row_end = Y.g < L.nyg ? min(L.n, Y.row_begin + L.ryg) : Y.row_begin;
  Y.nblk = (L.ryg + R - 1) / R;
  Y.f0 = Y.kl * L.yfc;
  Y.nf = max(0, min(L.F, Y.f0 + L.yfc) - Y.f0);
  Y.ps = Y.nf * a.W;
  const bool leader = Y.kl == 0;
  for (int j = 0; j < C::PT; ++j)
#pragma unroll
    for (int k = 0; k < RP; ++k) s_y[(j * RP + k) * kYThreads + threadIdx.x] = zero4();
  // every CTA of the cluster is running before any shared::cluster store
  cluster_arrive();
  cluster_wait();

  float pp[NV];
  y_phase1<RP>(a, L, Y, 0, pp);
  y_reduce_warps<RP>(pp, s_red[0]);
  __syncthreads();
  if (threadIdx.x < NV) y_push<RP>(Y, cw, s_red[0], s_slot[0]);
  cluster_arrive();
  double gacc = 0.0;  // leader, thread e < NG: Gram entry e of the group
  for (int b = 0; b < Y.nblk; ++b) {
    const int par = b & 1;
    const bool more = b + 1 < Y.nblk;
    if (more) {
      y_phase1<RP>(a, L, Y, b + 1, pp);
      y_reduce_warps<RP>(pp, s_red[par ^ 1]);
    }
    cluster_wait();  // block b's shares are in s_slot[par]
    __syncthreads();
    const int r0 = Y.row_begin + b * R;
    if (threadIdx.x < NV) {
      const int v = threadIdx.x;
      float s = 0.f;
      for (int q = 0; q < cw; ++q) s += s_slot[par][q * NV + v];
      s_prow[par][v] = s;
      const int row = r0 + v / RP;
      if (leader && row < Y.row_end) a.P[L.p_off + (int64_t)row * RP + v % RP] = s;
      // the members read block b - 1's shares before arriving for block b, and
      // every member has arrived for block b: s_slot[par ^ 1] is free
      if (more) y_push<RP>(Y, cw, s_red[par ^ 1], s_slot[par ^ 1]);
    }
    __syncthreads();
    if (leader && threadIdx.x < NG) {
      int i, j;
      tri_index(threadIdx.x, RP, i, j);
#pragma unroll
      for (int u = 0; u < R; ++u)
        if (r0 + u < Y.row_end) gacc = fma((double)s_prow[par][u * RP + i], (double)s_prow[par][u * RP + j], gacc);
    }
    y_phase2<RP>(a, L, Y, b, s_prow[par], s_y);
    if (more) cluster_arrive();
  }
  // no shared::cluster access follows: every store into this CTA's slots
  // preceded an arrival that the last wait covered
  if (Y.g >= L.nyg) return;
  float* yp = a.ypart + L.y_off + (int64_t)Y.g * a.W * L.ld * RP;
  for (int j = 0; j < C::PT; ++j) {
    const int p = (int)threadIdx.x + j * kYThreads;
    if (p >= Y.ps) break;
    const int w = p / Y.nf, f = Y.f0 + p % Y.nf;
    float4 y[RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) y[k] = s_y[(j * RP + k) * kYThreads + threadIdx.x];
    // element (column 4f + c, rank k) at (4f + c) * RP + k
    float4* dst = reinterpret_cast<float4*>(yp + (int64_t)w * L.ld * RP + (int64_t)(4 * f) * RP);
    if constexpr (RP == 1) {
      dst[0] = y[0];
    } else if constexpr (RP == 2) {
      dst[0] = make_float4(y[0].x, y[1].x, y[0].y, y[1].y);
      dst[1] = make_float4(y[0].z, y[1].z, y[0].w, y[1].w);
    } else {
      dst[0] = make_float4(y[0].x, y[1].x, y[2].x, y[3].x);
      dst[1] = make_float4(y[0].y, y[1].y, y[2].y, y[3].y);
      dst[2] = make_float4(y[0].z, y[1].z, y[2].z, y[3].z);
      dst[3] = make_float4(y[0].w, y[1].w, y[2].w, y[3].w);
    }
  }
  if (!leader) return;
  double* gp = a.gram + L.ygram_off;
  if (threadIdx.x < NG) gp[(int64_t)Y.g * NG + threadIdx.x] = gacc;
  gram_finish<RP>(a, L, gp, Y.g, L.nyg, a.counters + L.cnt_off + L.c_yg, s_gram, &s_flag, nullptr);
}

}  // namespace psgd
