// Combine: gate-weighted un-permute back to token order plus the shared
// experts' output, and two small utility kernels (weight packing, the bounded
// wait probe).
//
// y[t] = sum_{s kept} g~[t][s] * y_perm[slot_row[t][s]] + y_shared[t]
// ("MoE：条件计算与路由" §7 Eq.(3); the CSDN note's moe_infer un-permutes with
// new_x[idxs] = outs, then scales by topk_weight in fp32 and sums over k, and
// DeepseekV3MoE.forward adds shared_experts(identity)).  Dropped pairs
// (slot_row = -1) add nothing and the surviving gates are not renormalised
// (toy MoE demo).  One warp per token; fp32 accumulation in slot order, then
// the shared row; bf16 store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kCombineWarps = 8;

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4 v, float g) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
  }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

template <int K>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(int32_t T, int32_t d, const uint16_t* __restrict__ y_perm,
                   const int32_t* __restrict__ slot_row, const float* __restrict__ gates,
                   const uint16_t* __restrict__ y_shared, uint16_t* __restrict__ y, int64_t rmax,
                   int* status) {
  // vectors per lane per iteration: about 8 loads of 16 bytes in flight
  constexpr int U = (K + 1) >= 8 ? 1 : 8 / (K + 1);
  pdl_wait();  // y_perm (and y_shared) come from the down projection
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCombineWarps + warp;
  if (t >= T) return;
  int rows[K > 0 ? K : 1];
  float g[K > 0 ? K : 1];
#pragma unroll
  for (int s = 0; s < K; ++s) {
    rows[s] = slot_row[static_cast<int64_t>(t) * K + s];
    if (rows[s] >= 0 && !idx_ok(rows[s], rmax, status)) rows[s] = -1;
    g[s] = gates ? gates[static_cast<int64_t>(t) * K + s] : 1.0f;  // null: rows pre-scaled
  }
  const int nvec = d / 8;
  const uint4* ys = y_shared ? reinterpret_cast<const uint4*>(y_shared +
                                                              static_cast<int64_t>(t) * d)
                             : nullptr;
  uint4* out = reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * d);
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 val[U][K > 0 ? K : 1];
    uint4 sv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nvec) {
#pragma unroll
        for (int s = 0; s < K; ++s)
          if (rows[s] >= 0)
            val[u][s] = __ldg(reinterpret_cast<const uint4*>(
                                  y_perm + static_cast<int64_t>(rows[s]) * d) + v);
        if (ys) sv[u] = __ldg(ys + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) continue;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int s = 0; s < K; ++s)
        if (rows[s] >= 0) acc_bf16x8(acc, val[u][s], g[s]);
      if (ys) add_bf16x8(acc, sv[u]);
      out[v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// w13[g][2Mw][d]: 256-row block j = W1 rows [128j, 128j+128) then W3 rows.
__global__ void pack_w13_kernel(int32_t Mw, int32_t d, const uint16_t* __restrict__ w1,
                                const uint16_t* __restrict__ w3, uint16_t* __restrict__ w13) {
  const int64_t r = blockIdx.x;  // output row over G*2Mw
  const int64_t g = r / (2 * Mw);
  const int64_t rl = r % (2 * Mw);
  const int64_t j = rl / 256;
  const int64_t within = rl % 256;
  const uint16_t* src = (within < 128 ? w1 : w3) + (g * Mw + j * 128 + (within & 127)) * d;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(w13 + r * d);
  for (int v = threadIdx.x; v < d / 8; v += blockDim.x) d4[v] = s4[v];
}

// ALF-LB bias update ("MoE：条件计算与路由", ALF-LB: overloaded experts' bias
// goes down, underloaded experts' up, rate gamma, outside the backward pass):
// b_e <- b_e + gamma * sign(k T / E - n_e), sign(0) = 0, one fp32 rounding.
__global__ void alf_bias_update_kernel(int32_t E, int32_t T, int32_t k,
                                       const int32_t* __restrict__ counts, float gamma,
                                       float* __restrict__ bias) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const double diff = static_cast<double>(k) * T / E - static_cast<double>(counts[e]);
  const float step = diff > 0.0 ? gamma : (diff < 0.0 ? -gamma : 0.0f);
  bias[e] = bias[e] + step;
}

// Waits on a barrier that nothing signals; the bounded wait records a timeout
// in *status and the kernel returns normally.
__global__ void timeout_probe_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, timeout_ns, status, nullptr);
  __syncthreads();
}

}  // namespace

int launch_combine(int32_t T, int32_t d, int32_t k, const uint16_t* y_perm,
                   const int32_t* slot_row, const float* gates, const uint16_t* y_shared,
                   uint16_t* y, int64_t rmax, int* status, cudaStream_t stream, bool pdl) {
  if (T == 0) return 0;
  const int grid = (T + kCombineWarps - 1) / kCombineWarps;
  void (*kern)(int32_t, int32_t, const uint16_t*, const int32_t*, const float*, const uint16_t*,
               uint16_t*, int64_t, int*) = nullptr;
  switch (k) {
    case 0: kern = combine_kernel<0>; break;
    case 1: kern = combine_kernel<1>; break;
    case 2: kern = combine_kernel<2>; break;
    case 3: kern = combine_kernel<3>; break;
    case 4: kern = combine_kernel<4>; break;
    case 5: kern = combine_kernel<5>; break;
    case 6: kern = combine_kernel<6>; break;
    case 7: kern = combine_kernel<7>; break;
    case 8: kern = combine_kernel<8>; break;
    default: return -2;
  }
  if (launch_kernel(kern, dim3(grid), dim3(kCombineWarps * 32), 0, stream, pdl, 1u, T, d, y_perm,
                    slot_row, gates, y_shared, y, rmax, status) != cudaSuccess)
    return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_pack_w13(int32_t G, int32_t Mw, int32_t d, const uint16_t* w1, const uint16_t* w3,
                    uint16_t* w13, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(G) * 2 * Mw;
  if (rows == 0) return 0;
  if (rows > 0x7fffffffLL) return -2;
  pack_w13_kernel<<<static_cast<unsigned>(rows), 128, 0, stream>>>(Mw, d, w1, w3, w13);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_alf_bias_update(int32_t E, int32_t T, int32_t k, const int32_t* counts, float gamma,
                           float* bias, cudaStream_t stream) {
  alf_bias_update_kernel<<<(E + 255) / 256, 256, 0, stream>>>(E, T, k, counts, gamma, bias);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_timeout_probe(int* status, uint64_t timeout_ns, cudaStream_t stream) {
  timeout_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
