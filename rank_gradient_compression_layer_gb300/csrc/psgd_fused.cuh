// The fused step for padded ranks r <= 4: ONE launch per step that runs the
// tiles of all four phases (project, orthonormalise, back-project,
// decompress) from one queue.
//
// Why: on a model of many small layers (the ResNet-18 set) four phase
// launches leave the GPU draining at every phase boundary, and the
// back-project re-reads the error state B from HBM because the whole
// project phase has streamed past it.  Here a layer's back-project tiles run
// shortly after its project tiles, while its B is still in L2, and the
// phases of different layers overlap.
//
// How: the queue (built on the host, psgd_plan.h) lists every tile in an
// order where each tile's producers come first.  A CTA takes the next queue
// position with one atomic (a ticket), so positions are taken in order, and
// a tile whose inputs are not ready waits for a flag that the last CTA of
// the producing phase of that layer raises to the step's epoch:
//
//   project tiles  -> (the layer's last one stores R)        flag R
//   orthonormalise -> (the layer's last one stores X)        flag X
//   back-project   -> (each segment's last one stores Qbar)  flag Qbar[seg]
//   decompress     waits for Qbar[seg] and Qbar[0] (segment 0's tiles store
//                  the Phat rows it reads)
//
// A waiting CTA only ever waits on positions taken before its own, by CTAs
// that are running or done, so every wait ends.  Waits are still bounded
// (wait_ns, and an iteration cap): a wait that runs out marks the step as
// abandoned in sync[2], every CTA then stops taking work, and the host
// reports the failure at its next synchronising call.
//
// Data written by another CTA of this launch is read with ld.global.cg (L2;
// L1 is not coherent between SMs); see the FUSED variants of the bodies.
#pragma once

#include "psgd_kernels.cuh"

namespace psgd {

constexpr int kFThreads = 256;

template <int RP>
struct FusedCfg {
  static_assert(RP <= 4, "the fused step covers padded ranks 1, 2 and 4");
  // back-project rows per warp group: fewer than the phase kernel's, so the
  // whole step fits the register budget below (its B reads hit L2)
  static constexpr int UNR = RP <= 2 ? 8 : 4;
  static constexpr int MINB = 3;  // resident CTAs per SM the registers must allow
  static constexpr int RH = RP;                  // no rank split below r = 32
  // shared memory of each tile kind, in bytes; the CTA's buffer is the largest
  static constexpr size_t P_BYTES =
      (size_t)(kFThreads / 32) * Cfg<RP>::R1 * RP * 4 + (size_t)Cfg<RP>::R1 * RP * 4 + RP * RP * 8;
  static constexpr size_t H_BYTES = (size_t)(RP * RP + RP) * 8 + (size_t)ph_rows(RP) * RP * 4 + RP * RP * 8;
  static constexpr size_t B_BYTES = (size_t)(kFThreads / 32) * UNR * RH * 4 + RP * RP * 8 + p3_dyn_bytes(RP);
  static constexpr size_t U_BYTES = (size_t)Cfg<RP>::RU * RP * 4;
  static constexpr size_t cmax(size_t x, size_t y) { return x > y ? x : y; }
  static constexpr size_t SMEM = cmax(cmax(P_BYTES, H_BYTES), cmax(B_BYTES, U_BYTES));
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr unsigned kWaitMaxPolls = 1u << 22;  // a second cap on a wait, beside the time limit

// Whole CTA: wait until *f0 and *f1 (f1 may be null) hold this step's epoch.
// Thread 0 polls with acquire loads; the barrier then orders every thread's
// later reads after the producers' writes.  Returns false when the step was
// abandoned (this wait ran out, or another CTA's did).
static __device__ __noinline__ bool fused_wait(const StepArgs& a, const unsigned* f0, const unsigned* f1, int* s_ok) {
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint64_t t0 = global_timer_ns();
    for (unsigned it = 0;; ++it) {
      const unsigned v0 = ld_acquire_u32(f0);
      const unsigned v1 = f1 ? ld_acquire_u32(f1) : a.epoch;
      if ((int)(v0 - a.epoch) >= 0 && (int)(v1 - a.epoch) >= 0) break;
      if (ld_relaxed_u32(a.sync + 2) != 0u) {
        ok = 0;
        break;
      }
      if (it >= kWaitMaxPolls || (int64_t)(global_timer_ns() - t0) > a.wait_ns) {
        atomicCAS(a.sync + 2, 0u, 1u);
        ok = 0;
        break;
      }
      __nanosleep(it < 16 ? 32 : 256);
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// The tile bodies on the CTA's shared buffer.
template <int RP>
static __device__ __forceinline__ void fused_project(const StepArgs& a, const Tile& t, unsigned char* s_buf, int* s_flag,
                                                  unsigned* pub) {
  float* s_red = reinterpret_cast<float*>(s_buf);
  float* s_prow = s_red + (kFThreads / 32) * Cfg<RP>::R1 * RP;
  double* s_gram = reinterpret_cast<double*>(s_prow + Cfg<RP>::R1 * RP);
  p1_body<RP>(a, t, s_red, s_prow, s_gram, s_flag, pub);
}

template <int RP>
static __device__ __forceinline__ void fused_ortho(const StepArgs& a, const Tile& t, unsigned char* s_buf, int* s_flag,
                                                unsigned* pub) {
  double* s_r = reinterpret_cast<double*>(s_buf);
  double* s_gram = s_r + RP * RP + RP;
  float* s_p1 = reinterpret_cast<float*>(s_gram + RP * RP);
  ph_body<RP>(a, a.layers[t.layer], t.a, s_r, s_p1, s_gram, s_flag, pub);
}

template <int RP>
static __device__ __forceinline__ void fused_back(const StepArgs& a, const Tile& t, unsigned char* s_buf, int* s_flag,
                                               unsigned* pub) {
  using C = FusedCfg<RP>;
  float* s_red = reinterpret_cast<float*>(s_buf);  // p3_dyn_bytes, 16-byte aligned
  double* s_x = reinterpret_cast<double*>(s_red + p3_dyn_bytes(RP) / 4);
  float* s_ph = reinterpret_cast<float*>(s_x + RP * RP);
  const LayerDev L = a.layers[t.layer];  // by value: stores to B cannot alias it
  p3_body<RP, C::UNR, true>(a, t, L, s_ph, s_x, s_red, s_flag, pub);
}

template <int RP>
static __device__ __forceinline__ void fused_decomp(const StepArgs& a, const Tile& t, unsigned char* s_buf) {
  LayerDev L{};  // by value: stores to U cannot alias it (matrix tiles only)
  if (t.c != 1) L = a.layers[t.layer];
  u_body<RP, true>(a, t, L, reinterpret_cast<float*>(s_buf));
}

// Thread 0: the next queue position (n_items once the step was abandoned).
__device__ __forceinline__ int take_ticket(const StepArgs& a) {
  return ld_relaxed_u32(a.sync + 2) == 0u ? (int)atomicAdd(a.sync, 1u) : a.n_items;
}

template <int RP>
__global__ void __launch_bounds__(kFThreads, FusedCfg<RP>::MINB) fused_step_kernel(const StepArgs a) {
  __shared__ __align__(16) unsigned char s_buf[FusedCfg<RP>::SMEM];
  __shared__ int s_item[2];
  __shared__ int s_flag, s_ok;
  pdl_enter();
  int next = 0;  // thread 0: the position taken for the following iteration
  if (threadIdx.x == 0) s_item[0] = take_ticket(a);
  for (int iter = 0;; ++iter) {
    __syncthreads();  // s_item visible; every thread is done with the previous tile's shared memory
    const int idx = s_item[iter & 1];
    if (idx >= a.n_items) break;
    // the next position is taken now and used only after this tile, so the
    // atomic's round trip overlaps the tile (a CTA holding two positions
    // still runs them in order, and each depends on earlier ones only)
    if (threadIdx.x == 0) next = take_ticket(a);
    Tile t = a.tiles[idx];
    const int kind = t.layer >> kLayerBits;
    t.layer &= (1 << kLayerBits) - 1;
    if (kind == kItemDecomp && t.c == 1) {  // vector layer: no inputs from this step
      fused_decomp<RP>(a, t, s_buf);
    } else {
      unsigned* fl = a.flags + a.layers[t.layer].f_off;
      switch (kind) {
        case kItemProject:
          fused_project<RP>(a, t, s_buf, &s_flag, fl + kFlagR);
          break;
        case kItemOrtho:
          if (fused_wait(a, fl + kFlagR, nullptr, &s_ok)) fused_ortho<RP>(a, t, s_buf, &s_flag, fl + kFlagX);
          break;
        case kItemBack:
          if (fused_wait(a, fl + kFlagX, nullptr, &s_ok))
            fused_back<RP>(a, t, s_buf, &s_flag, fl + kFlagQbar + t.b);
          break;
        case kItemDecomp:
          if (fused_wait(a, fl + kFlagQbar + t.b, fl + kFlagQbar, &s_ok)) fused_decomp<RP>(a, t, s_buf);
          break;
        default:
          break;
      }
    }
    if (threadIdx.x == 0) s_item[(iter + 1) & 1] = next;
  }
  // the CTA takes no more work: the last one to get here resets the ticket
  // for the next step (no CTA of this launch takes a ticket after its own
  // last, failed one)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sync + 1, 1u) == gridDim.x - 1) {
      a.sync[0] = 0u;
      a.sync[1] = 0u;
    }
  }
}

}  // namespace psgd
