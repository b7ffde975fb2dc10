// rTop-k sparsification, the second compressor behind the C ABI (rTop-k
// review page, "rTop-k: A Statistical Estimation Approach to Distributed
// SGD", proposed method, bullet 3).  Host interface used by psgd_api.cu; the
// kernels and their planning live in psgd_rtopk.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "psgd_internal.h"

namespace psgd {

struct RTopK;

// Plans the selection of every (worker, matrix layer) problem of a layer set
// and allocates its device buffers.  hl / hv: the context's matrix and vector
// layer records (host copies); d_layers, d_vecs: their device copies.
int rtopk_create(RTopK** out, const std::vector<LayerDev>& hl, const std::vector<VecDev>& hv,
                 const LayerDev* d_layers, const VecDev* d_vecs, int W, uint64_t seed, int top_div,
                 int sample_div);
void rtopk_destroy(RTopK* rk);

// One step on stream s: M_w = G_w + E_w (E_w is B_w), the top set and the
// sampled subset of every problem, B_w <- M_w - S_w, the sparse messages,
// and U (matrix layers: (sum_w S_w) / W; vector layers: the worker mean)
// when U is not NULL.  step: the index of this step (for the draws).
// ev: NULL, or four events recorded after pass 0, pass 1, the tail and the
// apply (+ vector) kernels.
int rtopk_step(RTopK* rk, const float* const* G, float* B, int64_t total, float* U, int64_t step,
               cudaStream_t s, const cudaEvent_t* ev);

// k of matrix layer mi (its position among the matrix layers).
int64_t rtopk_k(const RTopK* rk, int mi);
// Device addresses of worker w's message for matrix layer mi: k indices
// (flat, row-major over n x m, ascending) and their k values.
void rtopk_message(const RTopK* rk, int mi, int w, const int32_t** idx, const float** val);
// Kernel launches one step enqueues.
int rtopk_launches(const RTopK* rk);
// Gathers every message of the last step into dst (device, rtopk_message_floats
// floats) in psgd_step_host's order: per matrix layer, per worker, its k
// indices (int32 bits) then its k values.  One kernel on stream s.
int rtopk_pack(const RTopK* rk, float* dst, cudaStream_t s);

}  // namespace psgd
