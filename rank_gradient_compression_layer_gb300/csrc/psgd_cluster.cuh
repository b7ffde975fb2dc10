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
// cluster of kYClusterMax CTAs holds S = kYClusterMax / cw such subgroups.
// The grid is persistent: one cluster per resident slot, each walking its own
// run of segments (a layer's consecutive blocks of R rows; subgroup s takes
// the segment's blocks s, s + S, ...), the runs cut for equal work.  Round i
// of a segment, per CTA:
//   1. for block i + 1: stream G and B of the slice (128-bit loads), rebuild
//      E = B - Phat' Q_w'^T, store M = G + E to B, and sum this CTA's share
//      of the block's P rows (warp butterfly, fixed-order sum over warps);
//      interleaved with the same loop, for block i - 1 (whose P rows are
//      known): re-read the M rows this thread stored two rounds before (L2
//      hits) and accumulate Y_w += M_w^T P in shared memory -- the HBM
//      stream and the L2 re-reads are in flight together;
//   2. wait on the cluster barrier for block i's shares (pushed into every
//      subgroup member's shared memory with st.shared::cluster, then a
//      release arrive), sum them in rank order -- every member gets the same
//      P rows, bit for bit -- and push block i + 1's share, arrive.
// The subgroup's first CTA stores the P rows and keeps float64 Gram sums.
// At the end of a segment the S subgroups' Y accumulators (same columns)
// and Gram sums are added in subgroup order through distributed shared
// memory, and the first subgroup stores the segment's Y partial (one slot)
// and runs the Gram tail (gram_finish) over the layer's slots.  The result
// does not depend on which cluster runs which segment.
#pragma once

#include "psgd_kernels.cuh"

namespace psgd {

template <int RP>
struct YCfg {
  static constexpr int R = y_rows(RP);         // rows of a block
  static constexpr int RU = 2;                 // rows whose loads are in flight together
  static constexpr int NV = R * RP;            // P values of a block
  static constexpr int NW = kYThreads / 32;
  static_assert(NV == 16, "a block's P values are one 16-value warp butterfly");
  static_assert(R % RU == 0, "whole chunks of rows");
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
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// The shared::cluster address of `local` in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, unsigned rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(const float* local, unsigned rank, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr(local, rank)), "f"(v) : "memory");
}

__device__ __forceinline__ float4 ld_cluster_f4(const float4* local, unsigned rank) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr(local, rank))
               : "memory");
  return v;
}

__device__ __forceinline__ double ld_cluster_f64(const double* local, unsigned rank) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(cluster_addr(local, rank)) : "memory");
  return v;
}

// The geometry of one CTA within a segment.
struct YTile {
  int sub, kl, S;           // subgroup, rank within it, subgroups of the cluster
  int b0, b1;               // the segment's blocks [b0, b1)
  int iters;                // rounds of S blocks (the same in the whole cluster)
  int f0, nf, ps;           // first float4 column, float4 columns and pairs of the slice
};

// The rows [r0, r1) of this subgroup's block in round i (empty outside the
// segment's rounds and past its blocks).
template <int RP>
__device__ __forceinline__ void y_block_rows(const LayerDev& L, const YTile& Y, int i, int& r0, int& r1) {
  const int blk = Y.b0 + Y.sub + i * Y.S;
  r0 = blk * L.yr;
  r1 = (i >= 0 && i < Y.iters && blk < Y.b1) ? min(L.n, r0 + L.yr) : r0;
}

// One pass over this thread's pairs: step 1 for the rows [n0, n1) (E, M
// stored to B, and this thread's share of their P values in pp[u * RP + k],
// row n0 + u, rank k) and Y += M[rows]^T P[rows] for the rows [o0, o1),
// whose P values are s_p (row o0 + u, rank k at u * RP + k).  s_y: RP float4
// per pair, pair p = thread + j kYThreads at (j RP + k) kYThreads + thread.
template <int RP>
__device__ __forceinline__ void y_pass(const StepArgs& a, const LayerDev& L, const YTile& Y, int n0, int n1,
                                       int o0, int o1, const float* s_p, float4* s_y, float (&pp)[YCfg<RP>::NV]) {
  using C = YCfg<RP>;
  constexpr int R = C::R, RU = C::RU;
#pragma unroll
  for (int i = 0; i < C::NV; ++i) pp[i] = 0.f;
  const bool ph1 = n0 < n1, ph2 = o0 < o1;
  if (!ph1 && !ph2) return;
  const bool prev = a.has_prev != 0;
  const float* Pprev = a.Phat + L.p_off + (int64_t)n0 * RP;
  for (int p = (int)threadIdx.x, j = 0; p < Y.ps; p += kYThreads, ++j) {
    const int w = p / Y.nf, f = Y.f0 + p % Y.nf;
    const float* Gw = a.G[w] + L.off + 4 * f;
    float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * f;
    // this pair's 4 rows of Q and of Q_w' (rows 4f .. 4f + 3 of ld x RP)
    float qv[4][RP], qw[4][RP];
    if (ph1) {
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
    float4 y[RP];
    if (ph2)
#pragma unroll
      for (int k = 0; k < RP; ++k) y[k] = s_y[(j * RP + k) * kYThreads + threadIdx.x];
    const bool tailc = (f == L.F - 1) && (L.tail < 4);
#pragma unroll
    for (int u0 = 0; u0 < R; u0 += RU) {
      if (n0 + u0 >= n1 && o0 + u0 >= o1) break;  // blocks of fewer than R rows
      float4 gv[RU], bv[RU], mv[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int row = n0 + u0 + u;
        if (row < n1) {
          gv[u] = __ldcs(reinterpret_cast<const float4*>(Gw + (int64_t)row * L.ld));
          bv[u] = __ldcs(reinterpret_cast<const float4*>(Bw + (int64_t)row * L.ld));
        } else {
          gv[u] = zero4();
          bv[u] = zero4();
        }
        const int orow = o0 + u0 + u;
        // this thread stored these M values two rounds before (program order)
        mv[u] = orow < o1 ? __ldcg(reinterpret_cast<const float4*>(Bw + (int64_t)orow * L.ld)) : zero4();
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int row = n0 + u0 + u;
        if (row < n1) {
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
          // a plain store: the line stays in L2 for the re-read two rounds on
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
        if (o0 + u0 + u < o1) {
#pragma unroll
          for (int k = 0; k < RP; ++k) {
            const float pv = s_p[(u0 + u) * RP + k];
            y[k].x = fmaf(mv[u].x, pv, y[k].x);
            y[k].y = fmaf(mv[u].y, pv, y[k].y);
            y[k].z = fmaf(mv[u].z, pv, y[k].z);
            y[k].w = fmaf(mv[u].w, pv, y[k].w);
          }
        }
      }
    }
    if (ph2)
#pragma unroll
      for (int k = 0; k < RP; ++k) s_y[(j * RP + k) * kYThreads + threadIdx.x] = y[k];
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

// Shared memory of the one-pass project kernel besides the Y accumulators.
template <int RP>
struct YShared {
  float slot[2][kYClusterMax * YCfg<RP>::NV];  // the subgroup's shares of a block's P values
  float red[2][YCfg<RP>::NW * YCfg<RP>::NV];   // the warps' shares
  float prow[3][YCfg<RP>::NV];                 // P values of the last three blocks
  double gacc[Cfg<RP>::NG];                    // the subgroup's Gram sums, at the end of a segment
  double gram[RP * RP];
  int flag;
};

// One segment of the cluster's run (every CTA of the cluster calls it).
template <int RP>
__device__ __forceinline__ void y_segment(const StepArgs& a, const Tile& sg, unsigned rank, float4* s_y,
                                          YShared<RP>& sh) {
  using C = YCfg<RP>;
  constexpr int NV = C::NV, NG = Cfg<RP>::NG, R = C::R;
  const LayerDev L = a.layers[sg.layer];  // by value: stores to B cannot alias it
  const int cw = L.cw;
  YTile Y;
  Y.S = kYClusterMax / cw;
  Y.sub = (int)rank / cw;
  Y.kl = (int)rank % cw;
  Y.b0 = sg.a;
  Y.b1 = sg.b;
  Y.iters = (sg.b - sg.a + Y.S - 1) / Y.S;
  Y.f0 = Y.kl * L.yfc;
  Y.nf = max(0, min(L.F, Y.f0 + L.yfc) - Y.f0);
  Y.ps = Y.nf * a.W;
  const bool leader = Y.kl == 0;
  // every CTA of the cluster is running, and done with the previous
  // segment's shared memory (slots, Y and Gram sums), before this one
  cluster_sync();
  for (int p = (int)threadIdx.x, j = 0; p < Y.ps; p += kYThreads, ++j)
#pragma unroll
    for (int k = 0; k < RP; ++k) s_y[(j * RP + k) * kYThreads + threadIdx.x] = zero4();

  float pp[NV];
  int r0, r1, n0, n1, o0, o1;
  y_block_rows<RP>(L, Y, 0, n0, n1);
  y_pass<RP>(a, L, Y, n0, n1, 0, 0, sh.prow[0], s_y, pp);
  y_reduce_warps<RP>(pp, sh.red[0]);
  __syncthreads();
  if (threadIdx.x < NV) y_push<RP>(Y, cw, sh.red[0], sh.slot[0]);
  cluster_arrive();
  double gacc = 0.0;  // leader, thread e < NG: Gram entry e of the subgroup's rows
  for (int i = 0; i < Y.iters; ++i) {
    const int par = i & 1;
    const bool more = i + 1 < Y.iters;
    y_block_rows<RP>(L, Y, i + 1, n0, n1);  // step 1 for the next block (empty in the last round)
    y_block_rows<RP>(L, Y, i - 1, o0, o1);  // Y for the block before (empty in the first round)
    y_pass<RP>(a, L, Y, n0, n1, o0, o1, sh.prow[(i + 2) % 3], s_y, pp);
    if (more) y_reduce_warps<RP>(pp, sh.red[par ^ 1]);
    cluster_wait();  // round i's shares are in slot[par]
    __syncthreads();
    y_block_rows<RP>(L, Y, i, r0, r1);
    if (threadIdx.x < NV) {
      const int v = threadIdx.x;
      float s = 0.f;
      for (int q = 0; q < cw; ++q) s += sh.slot[par][q * NV + v];
      sh.prow[i % 3][v] = s;
      const int row = r0 + v / RP;
      if (leader && row < r1) a.P[L.p_off + (int64_t)row * RP + v % RP] = s;
      // the members read round i - 1's shares before arriving for round i, and
      // every member has arrived for round i: slot[par ^ 1] is free
      if (more) y_push<RP>(Y, cw, sh.red[par ^ 1], sh.slot[par ^ 1]);
    }
    __syncthreads();
    if (leader && threadIdx.x < NG) {
      int ii, jj;
      tri_index(threadIdx.x, RP, ii, jj);
#pragma unroll
      for (int u = 0; u < R; ++u)
        if (r0 + u < r1) gacc = fma((double)sh.prow[i % 3][u * RP + ii], (double)sh.prow[i % 3][u * RP + jj], gacc);
    }
    if (more) cluster_arrive();
  }
  y_block_rows<RP>(L, Y, Y.iters - 1, o0, o1);
  y_pass<RP>(a, L, Y, 0, 0, o0, o1, sh.prow[(Y.iters - 1) % 3], s_y, pp);
  if (leader && threadIdx.x < NG) sh.gacc[threadIdx.x] = gacc;
  // every subgroup's Y and Gram sums are final
  cluster_sync();
  if (Y.sub != 0) return;
  // the first subgroup adds the other subgroups' sums (the same columns) in
  // subgroup order and stores the segment's slot
  const int slot = sg.c;
  float* yp = a.ypart + L.y_off + (int64_t)slot * a.W * L.ld * RP;
  for (int p = (int)threadIdx.x, j = 0; p < Y.ps; p += kYThreads, ++j) {
    const int w = p / Y.nf, f = Y.f0 + p % Y.nf;
    float4 y[RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) y[k] = s_y[(j * RP + k) * kYThreads + threadIdx.x];
    for (int s = 1; s < Y.S; ++s)
#pragma unroll
      for (int k = 0; k < RP; ++k) {
        const float4 o = ld_cluster_f4(s_y + (j * RP + k) * kYThreads + threadIdx.x, (unsigned)(s * cw + Y.kl));
        y[k].x += o.x;
        y[k].y += o.y;
        y[k].z += o.z;
        y[k].w += o.w;
      }
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
  if (threadIdx.x < NG) {
    double g = sh.gacc[threadIdx.x];
    for (int s = 1; s < Y.S; ++s) g += ld_cluster_f64(&sh.gacc[threadIdx.x], (unsigned)(s * cw));
    gp[(int64_t)slot * NG + threadIdx.x] = g;
  }
  gram_finish<RP>(a, L, gp, slot, L.nys, a.counters + L.cnt_off + L.c_yg, sh.gram, &sh.flag, nullptr);
}

// The persistent grid: cluster c runs the segments of header tile c.  Every
// CTA of a cluster runs the same segments and rounds, so the cluster barriers
// match; no CTA waits on another cluster.
template <int RP>
__global__ void __launch_bounds__(kYThreads, 2) p1c_kernel(const StepArgs a) {
  extern __shared__ float4 s_y[];  // the Y accumulators
  __shared__ YShared<RP> sh;
  pdl_enter();
  const Tile hdr = a.tiles[cluster_index()];
  const unsigned rank = cluster_ctarank();
  for (int si = 0; si < hdr.b; ++si) y_segment<RP>(a, a.tiles[a.y_clusters + hdr.a + si], rank, s_y, sh);
  // the first subgroup may still be reading this CTA's shared memory
  cluster_sync();
}

}  // namespace psgd
