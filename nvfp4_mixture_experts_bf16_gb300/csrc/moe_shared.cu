// moe_shared.cu — the shared expert of a layer: a BF16 SwiGLU expert scaled by a sigmoid gate.
//
// The model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix (bit-exact)", section "What is
// bit-exact and what is quantized", keeps the shared experts and the shared-expert gate in BF16
// and gives no formula; the Qwen-style form is taken. For token t:
//   sigma_t = 1 / (1 + exp(-x_t . gv)),   hs = BF16( SiLU(Wg x_t) * (Wu x_t) ),   Ys = Wd hs,
// all products exact BF16 x BF16 accumulated in FP32. Ys is stored in FP32 as computed; the
// combines round it to BF16 (an expert output, like the routed Y) and add sigma_t * BF16(Ys)
// after the routed terms, before the output's rounding.
//
// One or two tokens run the shared expert inside the fused narrow kernel (moe_decode.cu). Other
// narrow calls (T <= 8) are two CUDA-core GEMVs over the BF16 weights (6 MB gate/up, 3 MB down
// at H = 4096, Is = 384), one CTA per SM, each row read by one CTA with 16-byte loads on
// consecutive lanes; a CTA issues its first weight loads before waiting on the preceding
// kernel, so they stream while that kernel drains. Wide calls run the two products on the
// tcgen05 BF16 GEMM of the router (tensor cores: 2 T Is H FLOP each), with one per-token kernel
// in between for SiLU * up, the BF16 h and the gate.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kShThreads = 256;
constexpr int kShWarps = kShThreads / 32;
constexpr int kGuIdx = 3;               // intermediate indices per gate/up batch (2 rows each)
constexpr int kGuRows = 2 * kGuIdx;
constexpr int kGuUnits = 2;             // 16-byte units per lane and row of one K-chunk
constexpr int kGuChunk = kGuUnits * kShThreads;   // units of one K-chunk (4096 columns)
constexpr int kDnRows = 4;              // down rows per warp batch
constexpr int kDnUnits = 2;             // 16-byte units per lane and row kept in registers

__device__ __forceinline__ uint4 ldg128(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ldcg128(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

// Narrow gate/up: CTA b owns intermediate indices [j0, j1) of 0..Is, index Is being the gate
// vector. A batch holds kGuIdx indices (gate row, up row each); every warp takes an eighth of
// the 16-byte units of every row of the batch, K in chunks of kGuChunk units, so the CTA's 8
// warps cover each row once. With one token the kernel fits in 85 registers a thread,
// so its CTAs are resident next to the preceding narrow-call kernel's and their weight loads
// (issued before the wait) stream while that kernel runs.
template <int NT>
__global__ void __launch_bounds__(kShThreads, NT == 1 ? 3 : 1)
    k_shared_gu_narrow(const uint16_t* __restrict__ x, ShView sv, int H) {
  extern __shared__ __align__(16) unsigned char xs[];   // [NT][H] BF16
  __shared__ float red[kShWarps][kGuRows][NT];
  __shared__ float tot[kGuRows][NT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Is = sv.Is, nidx = Is + 1, G = gridDim.x, b = blockIdx.x;
  const int j0 = (int)((long long)nidx * b / G), j1 = (int)((long long)nidx * (b + 1) / G);
  const int nunits = H / 8, nkc = (nunits + kGuChunk - 1) / kGuChunk;
  uint4 w[kGuRows][kGuUnits];
  // row r of the batch at index jb: gate row (r even) or up row (r odd); the gate vector has
  // one row; absent rows load zeros
  auto load_batch = [&](int jb, int kc) {
#pragma unroll
    for (int r = 0; r < kGuRows; ++r) {
      const int j = jb + r / 2;
      const uint16_t* row = nullptr;
      if (j < j1) {
        if (j < Is) row = sv.gate_up + (size_t)(j + ((r & 1) ? Is : 0)) * H;
        else if ((r & 1) == 0) row = sv.gate;
      }
#pragma unroll
      for (int i = 0; i < kGuUnits; ++i) {
        const int u = kc * kGuChunk + warp * 32 + lane + i * kShThreads;
        w[r][i] = (row && u < nunits) ? ldg128(row + (size_t)u * 8) : make_uint4(0, 0, 0, 0);
      }
    }
  };
  if (j0 < j1) load_batch(j0, 0);   // before the wait: weights do not depend on earlier kernels
  pdl_wait();
  pdl_launch_dependents();
  for (int o = tid; o < NT * nunits; o += kShThreads)
    reinterpret_cast<uint4*>(xs)[o] = ldcg128(x + (size_t)o * 8);
  __syncthreads();
  for (int jb = j0; jb < j1; jb += kGuIdx) {
    float acc[kGuRows][NT];
#pragma unroll
    for (int r = 0; r < kGuRows; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[r][t] = 0.0f;
    for (int kc = 0; kc < nkc; ++kc) {
      if (jb != j0 || kc != 0) load_batch(jb, kc);
#pragma unroll
      for (int i = 0; i < kGuUnits; ++i) {
        const int u = kc * kGuChunk + warp * 32 + lane + i * kShThreads;
        if (u < nunits) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + ((size_t)t * nunits + u) * 16);
#pragma unroll
            for (int r = 0; r < kGuRows; ++r) acc[r][t] += dot8_bf16(w[r][i], xv);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kGuRows; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float v = acc[r][t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0) red[warp][r][t] = v;
      }
    __syncthreads();
    if (tid < kGuRows * NT) {
      const int r = tid / NT, t = tid % NT;
      float s = 0.0f;
#pragma unroll
      for (int q = 0; q < kShWarps; ++q) s += red[q][r][t];
      tot[r][t] = s;
    }
    __syncthreads();
    if (tid < kGuIdx * NT) {
      const int q = tid / NT, t = tid % NT, j = jb + q;
      if (j < j1) {
        if (j < Is) {
          sv.hs[(size_t)t * Is + j] = f32_to_bf16_rn(silu_mul(tot[2 * q][t], tot[2 * q + 1][t]));
        } else {
          sv.sigma[t] = 1.0f / (1.0f + expf(-tot[2 * q][t]));
        }
      }
    }
  }
}

// Narrow down: CTA b owns output rows [r0, r1) of H; warp w takes rows r0 + w + 8 i in batches
// of kDnRows; lanes stride over a row's 16-byte units (the first kDnUnits per lane held in
// registers, loaded for the first batch before the wait).
template <int NT>
__global__ void __launch_bounds__(kShThreads, 1)
    k_shared_dn_narrow(ShView sv, int H) {
  extern __shared__ __align__(16) unsigned char hsm[];   // [NT][Is] BF16
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Is = sv.Is, G = gridDim.x, b = blockIdx.x;
  const int r0 = (int)((long long)H * b / G), r1 = (int)((long long)H * (b + 1) / G);
  const int nrw = (r1 - r0 > warp) ? (r1 - r0 - warp + kShWarps - 1) / kShWarps : 0;
  const int nu = Is / 8;
  uint4 w[kDnRows][kDnUnits];
  auto load_batch = [&](int rb) {
#pragma unroll
    for (int rr = 0; rr < kDnRows; ++rr) {
      const bool valid = rb + rr < nrw;
      const uint16_t* row = sv.down + (size_t)(r0 + warp + kShWarps * (rb + rr)) * Is;
#pragma unroll
      for (int c = 0; c < kDnUnits; ++c) {
        const int u = lane + 32 * c;
        w[rr][c] = (valid && u < nu) ? ldg128(row + (size_t)u * 8) : make_uint4(0, 0, 0, 0);
      }
    }
  };
  if (nrw > 0) load_batch(0);
  pdl_wait();
  pdl_launch_dependents();
  for (int o = tid; o < NT * nu; o += kShThreads)
    reinterpret_cast<uint4*>(hsm)[o] = ldcg128(sv.hs + (size_t)o * 8);
  __syncthreads();
  for (int rb = 0; rb < nrw; rb += kDnRows) {
    if (rb > 0) load_batch(rb);
    float acc[kDnRows][NT];
#pragma unroll
    for (int rr = 0; rr < kDnRows; ++rr)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[rr][t] = 0.0f;
#pragma unroll
    for (int c = 0; c < kDnUnits; ++c) {
      const int u = lane + 32 * c;
      if (u < nu) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 hv = *reinterpret_cast<const uint4*>(hsm + ((size_t)t * nu + u) * 16);
#pragma unroll
          for (int rr = 0; rr < kDnRows; ++rr) acc[rr][t] += dot8_bf16(w[rr][c], hv);
        }
      }
    }
    // units past the register-held ones (Is > 512)
    for (int u = 32 * kDnUnits + lane; u < nu; u += 32) {
#pragma unroll
      for (int rr = 0; rr < kDnRows; ++rr) {
        if (rb + rr < nrw) {
          const uint4 wv =
              ldg128(sv.down + (size_t)(r0 + warp + kShWarps * (rb + rr)) * Is + (size_t)u * 8);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            acc[rr][t] += dot8_bf16(wv, *reinterpret_cast<const uint4*>(hsm + ((size_t)t * nu + u) * 16));
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < kDnRows; ++rr) {
      const int row = r0 + warp + kShWarps * (rb + rr);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float v = acc[rr][t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == t && rb + rr < nrw) sv.ys[(size_t)t * H + row] = v;
      }
    }
  }
}

// Wide calls, between the two GEMMs: one CTA per token. h_j = BF16(SiLU(g_j) * u_j) from the
// FP32 products, and sigma_t from x_t . gv (8-product chunks, then a fixed-order tree).
__global__ void __launch_bounds__(kShThreads)
    k_shared_act_wide(const uint16_t* __restrict__ x, ShView sv, int T, int H) {
  __shared__ float part[kShThreads];
  const int t = blockIdx.x, tid = threadIdx.x, Is = sv.Is;
  pdl_wait();
  pdl_launch_dependents();
  if (t >= T) return;
  const float* gu = sv.gu + (size_t)t * 2 * Is;
  for (int j = tid; j < Is; j += kShThreads)
    sv.hs[(size_t)t * Is + j] = f32_to_bf16_rn(silu_mul(__ldcg(gu + j), __ldcg(gu + Is + j)));
  float a = 0.0f;
  for (int u = tid; u < H / 8; u += kShThreads)
    a += dot8_bf16(ldcg128(x + (size_t)t * H + (size_t)u * 8), ldg128(sv.gate + (size_t)u * 8));
  part[tid] = a;
  __syncthreads();
  for (int n = kShThreads / 2; n > 0; n >>= 1) {
    if (tid < n) part[tid] += part[tid + n];
    __syncthreads();
  }
  if (tid == 0) sv.sigma[t] = 1.0f / (1.0f + expf(-part[0]));
}


template <int NT>
cudaError_t launch_narrow(const LaunchCfg& lc, const uint16_t* x, const ShView& sv, int H) {
  const size_t xs_bytes = (size_t)NT * H * 2, hs_bytes = (size_t)NT * sv.Is * 2;
  cudaError_t e = cudaFuncSetAttribute(k_shared_gu_narrow<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xs_bytes);
  if (e != cudaSuccess) return e;
  const int gu_grid = lc.num_sms < sv.Is + 1 ? lc.num_sms : sv.Is + 1;
  e = launch_kernel(lc, k_shared_gu_narrow<NT>, dim3(gu_grid), dim3(kShThreads), xs_bytes, x, sv, H);
  if (e != cudaSuccess) return e;
  const int dn_grid = lc.num_sms < H ? lc.num_sms : H;
  return launch_kernel(lc, k_shared_dn_narrow<NT>, dim3(dn_grid), dim3(kShThreads), hs_bytes, sv, H);
}

}  // namespace

cudaError_t launch_shared(const LaunchCfg& lc, const uint16_t* x, const ShView& sv,
                          const WsView& ws, int* launches) {
  const int T = ws.T, H = ws.H;
  if (T <= kNarrowT) {
    if (launches) *launches += 2;
    switch (T) {
      case 1: return launch_narrow<1>(lc, x, sv, H);
      case 2: return launch_narrow<2>(lc, x, sv, H);
      case 3: return launch_narrow<3>(lc, x, sv, H);
      case 4: return launch_narrow<4>(lc, x, sv, H);
      case 5: return launch_narrow<5>(lc, x, sv, H);
      case 6: return launch_narrow<6>(lc, x, sv, H);
      case 7: return launch_narrow<7>(lc, x, sv, H);
      case 8: return launch_narrow<8>(lc, x, sv, H);
    }
    return cudaErrorInvalidValue;
  }
  if (!tc_supported()) return cudaErrorNotSupported;
  // gate/up: [T][2 Is] = x [T][H] . Wgu [2 Is][H]^T
  WsView g = ws;
  g.E = 2 * sv.Is;
  g.logits = sv.gu;
  cudaError_t e = launch_tc_router(lc, x, sv.gate_up, g);
  if (e != cudaSuccess) return e;
  e = launch_kernel(lc, k_shared_act_wide, dim3(T), dim3(kShThreads), 0, x, sv, T, H);
  if (e != cudaSuccess) return e;
  // down: [T][H] = hs [T][Is] . Wd [H][Is]^T
  WsView d = ws;
  d.H = sv.Is;
  d.E = H;
  d.logits = sv.ys;
  e = launch_tc_router(lc, sv.hs, sv.down, d);
  if (launches) *launches += 3;
  return e;
}

}  // namespace moe
