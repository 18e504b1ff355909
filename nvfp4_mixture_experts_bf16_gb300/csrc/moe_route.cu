// moe_route.cu — router, top-k + softmax, histogram + permutation, and activation preparation
// for the NVFP4 routed-expert MoE step (sm_103a).
//
// Model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix (bit-exact)": the router is stored
// BF16 and each token keeps the top-10 of 512 routed experts. Weights are the softmax over the
// selected logits; ties go to the lower expert index.
//
// Narrow calls (T <= 8, the decode / speculative-verification case of the Infernix release
// notes "windows-2026.10.11", "Highlights") run in ONE kernel: every CTA computes 4 router rows
// (a GEMV: the 4 MiB router is read once, coalesced) and prepares its share of the activations;
// the last CTA to finish (a ticket, no spinning) selects the top-k, the softmax weights, the
// histogram, the permutation and the token groups. Wide calls (prefill) run a tensor-core
// router GEMM followed by small top-k / histogram / scan / scatter kernels.
#include "moe_internal.cuh"

#include <cuda_bf16.h>
#include <float.h>

namespace moe {
namespace {

struct RouteOut {
  int32_t* idx;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
};

// Prepare one 16-element block of token t: the f16 B operand (and the W4A4 codes/scales).
__device__ __forceinline__ void prep_block(const uint16_t* xrow, int b, int t, const WsView& ws,
                                           int mode, float xS, float x_inv6S, int shift) {
  const int H = ws.H;
  const uint4* src = reinterpret_cast<const uint4*>(xrow + b * 16);
  const uint4 u0 = src[0], u1 = src[1];
  const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(words[i]);
    v[2 * i + 1] = bf16_hi(words[i]);
  }
  __half hv[16];
  if (mode == 0) {
    const float f = pow2f(-shift);
#pragma unroll
    for (int i = 0; i < 16; ++i) hv[i] = __float2half_rn(__fmul_rn(v[i], f));
  } else {
    uint32_t codes[2];
    const uint32_t sf = quantize16(v, xS, x_inv6S, codes);
    *reinterpret_cast<uint2*>(ws.xq + (size_t)t * (H / 2) + b * 8) = make_uint2(codes[0], codes[1]);
    ws.xsf[(size_t)t * (H / 16) + b] = static_cast<uint8_t>(sf);
    const float sfv = e4m3_value_nonneg(sf);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      hv[i] = __float2half_rn(e2m1_value((codes[i >> 3] >> (4 * (i & 7))) & 0xF) * sfv);
  }
  // permuted inside each 128-wide k-block: element 128J + 32c + 8p + q is stored at
  // 128J + 32p + 8c + q, so that the expert kernels read a thread's 32 values as 4 x 16 B
  const int J = b >> 3, c = (b & 7) >> 1, p0 = 2 * (b & 1);
  __half* row = ws.xh + (size_t)t * H + J * 128 + 8 * c;
  *reinterpret_cast<uint4*>(row + 32 * p0) = *reinterpret_cast<uint4*>(&hv[0]);
  *reinterpret_cast<uint4*>(row + 32 * (p0 + 1)) = *reinterpret_cast<uint4*>(&hv[8]);
}

// Block-wide exclusive scan of n <= 4 * blockDim ints in shared memory (in place); returns
// the total. blockDim.x must be 256.
__device__ int block_exclusive_scan(int32_t* a, int n, int32_t* scratch /*[8]*/) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int v[4], s = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = tid * 4 + i;
    v[i] = idx < n ? a[idx] : 0;
    s += v[i];
  }
  int incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  int wbase = 0, total = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) wbase += scratch[w];
    total += scratch[w];
  }
  int run = wbase + incl - s;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = tid * 4 + i;
    if (idx < n) a[idx] = run;
    run += v[i];
  }
  __syncthreads();
  return total;
}

// ------------------------------------------------------------------ narrow router
constexpr int kRouteRows = 4;  // router rows per CTA (2 warps per row, one per half of H)

// Fill the record of group u (expert e, slots [slot0, slot0 + n)); pk may be null (routing only).
__device__ __forceinline__ void write_group(const WsView& ws, const PackView* pk, int u, int e,
                                            int slot0, int n, const int32_t* perm_s) {
  GroupMeta m;
  m.expert = e;
  m.slot0 = slot0;
  m.n = n;
  m.pad0 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m.tok[i] = (perm_s && i < n) ? perm_s[slot0 + i] : -1;
  if (pk) {
    m.mg = pk->mult[e * 3 + 0];
    m.mu = pk->mult[e * 3 + 1];
    m.md = pk->mult[e * 3 + 2];
    m.sd = pk->down_in_scale[e];
    m.i6d = pk->down_inv6S[e];
  } else {
    m.mg = m.mu = m.md = m.sd = m.i6d = 0.0f;
  }
  m.pad1 = m.pad2 = m.pad3 = 0.0f;
  ws.gmeta[u] = m;
}

template <int NT>
__global__ void __launch_bounds__(256) k_route_narrow(const uint16_t* __restrict__ x,
                                                      const uint16_t* __restrict__ wr, WsView ws,
                                                      PackView pkv, int has_pack, int mode,
                                                      float xS, float x_inv6S, RouteOut out) {
  const PackView* pk = has_pack ? &pkv : nullptr;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float part[kRouteRows][2][kNarrowT];
  __shared__ int shift_s[kNarrowT];
  __shared__ int last_s;
  __shared__ int32_t scan_scratch[8];
  __shared__ uint64_t bar;

  const int T = NT, H = ws.H, E = ws.E, k = ws.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                       // [NT][H]
  const uint16_t* wrs = reinterpret_cast<const uint16_t*>(smem + (size_t)NT * H * 2);  // [4][H]
  const int row0 = blockIdx.x * kRouteRows;
  const int nrows = min(kRouteRows, E - row0);

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  // Two TMA bulk copies: the activations and this CTA's router rows (contiguous).
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)(NT + nrows) * H * 2);
    bulk_g2s(xs, x, (uint32_t)NT * H * 2, &bar);
    bulk_g2s(const_cast<uint16_t*>(wrs), wr + (size_t)row0 * H, (uint32_t)nrows * H * 2, &bar);
  }
  if (!mbar_wait(&bar, 0)) record_status(ws.ctl, kStTimeout);

  const int r = warp >> 1, half = warp & 1;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
  if (r < nrows) {
    const uint4* wrow = reinterpret_cast<const uint4*>(wrs + (size_t)r * H) + half * (H / 16);
    const int nchunk = H / 16;  // uint4 chunks in half a row
#pragma unroll 2
    for (int i = lane; i < nchunk; i += 32) {
      const uint4 wv = wrow[i];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint4 xv = reinterpret_cast<const uint4*>(xs + (size_t)t * H)[half * nchunk + i];
        acc[t] += dot8_bf16(wv, xv);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], off);
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t) part[r][half][t] = acc[t];
  }

  // Per-token power-of-two shift of the f16 operand (W4A16): one warp per token.
  if (mode == 0 && warp < T) {
    float m = 0.0f;
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs + (size_t)warp * H);
    for (int i = lane; i < H / 2; i += 32) {
      const uint32_t v = xr[i];
      m = fmaxf(m, fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) shift_s[warp] = token_shift(m);
  }
  __syncthreads();

  if (tid < kRouteRows * T) {
    const int rl = tid / T, t = tid % T;
    const int rr = row0 + rl;
    if (rr < E) ws.logits[(size_t)t * E + rr] = part[rl][0][t] + part[rl][1][t];
  }

  // This CTA's share of the activation preparation (skipped for routing-only calls).
  if (mode >= 0) {
    const int nblk = T * (H / 16);
    for (int it = blockIdx.x * 256 + tid; it < nblk; it += gridDim.x * 256) {
      const int t = it / (H / 16), b = it % (H / 16);
      prep_block(xs + (size_t)t * H, b, t, ws, mode, xS, x_inv6S, mode == 0 ? shift_s[t] : 0);
    }
    if (blockIdx.x == 0 && tid < T) ws.xfac[tid] = mode == 0 ? pow2f(shift_s[tid]) : xS;
  }

  // Last CTA to arrive finishes the routing.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t ticket = atomicAdd(&ws.ctl[kCtlRouteTicket], 1u);
    last_s = (ticket == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();

  const int S = T * k;
  int32_t* sel_idx = reinterpret_cast<int32_t*>(smem);                // [S]
  float* sel_w = reinterpret_cast<float*>(sel_idx + S);               // [S]
  int32_t* cnt = reinterpret_cast<int32_t*>(sel_w + S);               // [E+1]
  int32_t* uq = cnt + (E + 1);                                        // [E+1]
  uint32_t* tmask = reinterpret_cast<uint32_t*>(uq + (E + 1));        // [E] tokens per expert
  int32_t* perm_s = reinterpret_cast<int32_t*>(tmask + E);            // [S]

  for (int e = tid; e <= E; e += 256) {
    cnt[e] = 0;
    if (e < E) tmask[e] = 0u;
  }
  if (warp < T) {
    int e_sel;
    float w_sel;
    topk_row(ws.logits + (size_t)warp * E, E, k, lane, e_sel, w_sel);
    if (lane < k) {
      sel_idx[warp * k + lane] = e_sel;
      sel_w[warp * k + lane] = w_sel;
    }
  }
  __syncthreads();
  if (tid < S) {
    atomicAdd(&cnt[sel_idx[tid]], 1);
    atomicOr(&tmask[sel_idx[tid]], 1u << (tid / k));
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    uq[e] = cnt[e] > 0 ? 1 : 0;
    out.counts[e] = cnt[e];
    ws.counts[e] = cnt[e];
  }
  __syncthreads();
  block_exclusive_scan(cnt, E, scan_scratch);   // cnt -> offsets
  const int U = block_exclusive_scan(uq, E, scan_scratch);
  for (int e = tid; e < E; e += 256) {
    out.offsets[e] = cnt[e];
    ws.offsets[e] = cnt[e];
  }
  if (tid == 0) {
    out.offsets[E] = S;
    ws.offsets[E] = S;
    ws.ctl[kCtlGroups] = U;
    ws.ctl[kCtlUnique] = U;
  }
  if (tid < S) {
    // a token selects an expert at most once: its rank among the expert's slots is the number
    // of earlier tokens that selected the same expert
    const int t = tid / k, e = sel_idx[tid];
    const int pos = cnt[e] + __popc(tmask[e] & ((1u << t) - 1u));
    perm_s[pos] = t;
    out.perm[pos] = t;
    ws.perm[pos] = t;
    ws.slot_of[tid] = pos;
    out.idx[tid] = e;
    out.w[tid] = sel_w[tid];
    ws.idx[tid] = e;
    ws.w[tid] = sel_w[tid];
    if (ws.slot_amax) ws.slot_amax[tid] = 0u;
  }
  __syncthreads();
  // one group per distinct expert (a narrow call has at most 8 tokens per expert)
  for (int e = tid; e < E; e += 256) {
    const int c = ((e + 1 < E) ? cnt[e + 1] : S) - cnt[e];
    if (c > 0) {
      const int u = uq[e];
      write_group(ws, pk, u, e, cnt[e], c, perm_s);
    }
  }
  if (tid == 0) ws.ctl[kCtlRouteTicket] = 0u;
}

// ------------------------------------------------------------------ wide router GEMM
// logits[T][E] = x[T][H] . Wr[E][H]^T, BF16 mma.sync m16n8k16 with FP32 accumulation.
// CTA tile 128 tokens x 128 experts, k-step 32, two cp.async stages.
constexpr int kGM = 128, kGN = 128, kGK = 32, kGLd = 40;  // padded row (bf16 elements)

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool pred) {
  const uint32_t d = smem_u32(dst);
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(256) k_router_gemm(const uint16_t* __restrict__ x,
                                                     const uint16_t* __restrict__ wr, WsView ws) {
  __shared__ __align__(16) uint16_t As[2][kGM][kGLd];
  __shared__ __align__(16) uint16_t Bs[2][kGN][kGLd];
  const int T = ws.T, H = ws.H, E = ws.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m0 = blockIdx.y * kGM, n0 = blockIdx.x * kGN;
  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 64;  // warp tile 32 x 64

  pdl_wait();
  pdl_launch_dependents();

  auto load_stage = [&](int st, int k0) {
    // 128 rows x 32 bf16 = 512 chunks of 16 B per operand; 2 per thread per operand.
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + 256 * i, r = c >> 2, q = c & 3;
      const bool pa = (m0 + r) < T;
      const bool pb = (n0 + r) < E;
      cp_async16(&As[st][r][q * 8], x + (size_t)(pa ? m0 + r : 0) * H + k0 + q * 8, pa);
      cp_async16(&Bs[st][r][q * 8], wr + (size_t)(pb ? n0 + r : 0) * H + k0 + q * 8, pb);
    }
    cp_async_commit();
  };

  float acc[2][8][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.0f;

  const int nk = H / kGK;
  load_stage(0, 0);
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait_all();
    __syncthreads();
    if (kt + 1 < nk) load_stage((kt + 1) & 1, (kt + 1) * kGK);
    const int st = kt & 1;
#pragma unroll
    for (int kk = 0; kk < kGK; kk += 16) {
      uint32_t a[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = wm + i * 16 + (lane & 15);
        const int c = kk + (lane >> 4) * 8;
        ldmatrix_x4(a[i], &As[st][r][c]);
      }
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        uint32_t b[4];
        // matrices: (n j, k lo), (n j, k hi), (n j+1, k lo), (n j+1, k hi)
        const int r = wn + j * 8 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kk + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(b, &Bs[st][r][c]);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          mma_bf16_16816(acc[i][j], a[i], b[0], b[1]);
          mma_bf16_16816(acc[i][j + 1], a[i], b[2], b[3]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = m0 + wm + i * 16 + (lane >> 2);
      const int c = n0 + wn + j * 8 + (lane & 3) * 2;
      if (c + 1 < E + 1) {
        if (r < T && c < E) ws.logits[(size_t)r * E + c] = acc[i][j][0];
        if (r < T && c + 1 < E) ws.logits[(size_t)r * E + c + 1] = acc[i][j][1];
        if (r + 8 < T && c < E) ws.logits[(size_t)(r + 8) * E + c] = acc[i][j][2];
        if (r + 8 < T && c + 1 < E) ws.logits[(size_t)(r + 8) * E + c + 1] = acc[i][j][3];
      }
    }
}

// ------------------------------------------------------------------ wide top-k + histogram
constexpr int kChunkTok = 32;

// One block per chunk of 32 tokens, one warp per token: the top-k + softmax of the token, then
// the chunk's per-expert counts (its row of chunk_base, scanned into prefixes by k_scan_wide)
// and each selection's rank among the chunk's earlier selections of its expert (a token selects
// an expert at most once, so the rank is the number of earlier tokens in the chunk that
// selected it: a popcount of the expert's token mask), kept in slot_of for k_scatter_wide.
__global__ void __launch_bounds__(32 * kChunkTok) k_topk_wide(WsView ws, RouteOut out) {
  extern __shared__ __align__(16) unsigned char smem[];
  int32_t* cnt = reinterpret_cast<int32_t*>(smem);                  // [E]
  uint32_t* tmask = reinterpret_cast<uint32_t*>(cnt + ws.E);        // [E]: tokens of the chunk
  __shared__ unsigned long long cand[kChunkTok][32];   // per-warp selection scratch
  const int E = ws.E, k = ws.k, T = ws.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    cnt[e] = 0;
    tmask[e] = 0u;
  }
  __syncthreads();
  const int t = blockIdx.x * kChunkTok + warp;
  int e_sel = 0;
  if (t < T) {
    float w_sel;
    topk_row_scratch(ws.logits + (size_t)t * E, E, k, lane, cand[warp], e_sel, w_sel);
    if (lane < k) {
      out.idx[(size_t)t * k + lane] = e_sel;
      out.w[(size_t)t * k + lane] = w_sel;
      ws.idx[(size_t)t * k + lane] = e_sel;
      ws.w[(size_t)t * k + lane] = w_sel;
      atomicAdd(&cnt[e_sel], 1);
      atomicOr(&tmask[e_sel], 1u << warp);
    }
  }
  __syncthreads();
  if (t < T && lane < k)
    ws.slot_of[(size_t)t * k + lane] = __popc(tmask[e_sel] & ((1u << warp) - 1u));
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    ws.chunk_base[(size_t)blockIdx.x * E + e] = cnt[e];
}

// One CTA of 1024 threads: per-expert chunk prefix sums, offsets, and the token groups.
__global__ void __launch_bounds__(1024) k_scan_wide(WsView ws, PackView pkv, int has_pack,
                                                    RouteOut out, int nchunk) {
  const PackView* pk = has_pack ? &pkv : nullptr;
  __shared__ int32_t tot[1024 + 1];
  __shared__ int32_t wsum[32];
  __shared__ int32_t gsum[32][33];
  __shared__ int last_s;
  const int E = ws.E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  pdl_launch_dependents();
  {
    // this block's 32 experts (lane) x 32 groups of consecutive chunks (warp): the chunk counts
    // of each expert become its chunk prefixes in place (loads of a warp: 32 consecutive
    // experts of one chunk, 128 contiguous bytes)
    const int ec = blockIdx.x * 32 + lane;
    const int cpg = (nchunk + 31) / 32;
    const int c0 = warp * cpg, c1 = min(c0 + cpg, nchunk);
    int32_t* col = ws.chunk_base + ec;
    int mine = 0;
    if (ec < E)
      for (int c = c0; c < c1; ++c) mine += col[(size_t)c * E];
    gsum[warp][lane] = mine;
    __syncthreads();
    int run = 0;
    for (int w = 0; w < warp; ++w) run += gsum[w][lane];
    if (ec < E) {
      for (int c = c0; c < c1; ++c) {
        const int v = col[(size_t)c * E];
        col[(size_t)c * E] = run;
        run += v;
      }
      if (warp == 31) ws.counts[ec] = run;   // the expert's total
    }
  }
  // the last block to finish forms the offsets, groups and token tiles of every expert
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    last_s = atomicAdd(&ws.ctl[kCtlRouteTicket], 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  const int e = threadIdx.x;
  const int cnt_e = e < E ? __ldcg(&ws.counts[e]) : 0;
  const int ng_e = (cnt_e + kGroup - 1) / kGroup;
  const int nt_e = (cnt_e + 127) / 128;
  // three block-wide exclusive scans: slots, token groups, 128-slot token tiles
  int a = cnt_e, b = ng_e, c3 = nt_e;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int oa = __shfl_up_sync(0xFFFFFFFFu, a, off);
    const int ob = __shfl_up_sync(0xFFFFFFFFu, b, off);
    const int oc = __shfl_up_sync(0xFFFFFFFFu, c3, off);
    if (lane >= off) { a += oa; b += ob; c3 += oc; }
  }
  __shared__ int32_t tsum[32];
  if (lane == 31) { wsum[warp] = a; tot[warp] = b; tsum[warp] = c3; }
  __syncthreads();
  int ba = 0, bb = 0, bc = 0, ta = 0, tb = 0, tc = 0;
  for (int w = 0; w < 32; ++w) {
    if (w < warp) { ba += wsum[w]; bb += tot[w]; bc += tsum[w]; }
    ta += wsum[w];
    tb += tot[w];
    tc += tsum[w];
  }
  const int off_e = ba + a - cnt_e;
  const int gbase = bb + b - ng_e;
  const int tbase = bc + c3 - nt_e;
  __syncthreads();
  if (e < E) {
    out.counts[e] = cnt_e;
    out.offsets[e] = off_e;
    ws.counts[e] = cnt_e;
    ws.offsets[e] = off_e;
    // token groups of <= 8 slots feed the mma.sync expert kernels; the tensor-core path
    // reads the 128-slot token tiles instead
    if (!ws.tt_expert)
      for (int q = 0; q < ng_e; ++q)
        write_group(ws, pk, gbase + q, e, off_e + q * kGroup, min(kGroup, cnt_e - q * kGroup),
                    nullptr);
    if (ws.tt_expert) {
      ws.ttbase[e] = tbase;
      for (int q = 0; q < nt_e; ++q) {
        ws.tt_expert[tbase + q] = e;
        ws.tt_slot0[tbase + q] = off_e + q * 128;
        ws.tt_n[tbase + q] = min(128, cnt_e - q * 128);
      }
    }
  }
  if (e == 0) {
    if (ws.tt_expert) ws.ttbase[E] = tc;
    ws.ctl[kCtlTokenTiles] = tc;
  }
  if (ws.slot_amax)
    for (int i = e; i < ws.T * ws.k; i += 1024) ws.slot_amax[i] = 0u;
  if (e == 0) {
    out.offsets[E] = ta;
    ws.offsets[E] = ta;
    ws.ctl[kCtlGroups] = tb;
    ws.ctl[kCtlRouteTicket] = 0u;
  }
}

// Slot s = t*k + j of every token: its position in the expert-major permutation, from the
// expert's offset, the chunk's prefix for the expert and the selection's rank in the chunk.
__global__ void __launch_bounds__(256) k_scatter_wide(WsView ws, RouteOut out) {
  const int E = ws.E, k = ws.k;
  pdl_wait();
  pdl_launch_dependents();
  const int s = blockIdx.x * 256 + threadIdx.x;
  if (s >= ws.T * k) return;
  const int t = s / k, e = ws.idx[s];
  const int pos = ws.offsets[e] + ws.chunk_base[(size_t)(t / kChunkTok) * E + e] + ws.slot_of[s];
  out.perm[pos] = t;
  ws.perm[pos] = t;
  ws.slot_of[s] = pos;
}

// ------------------------------------------------------------------ wide activation prep
__global__ void __launch_bounds__(256) k_xprep_wide(const uint16_t* __restrict__ x, WsView ws,
                                                    int mode, float xS, float x_inv6S) {
  __shared__ float red[8];
  const int H = ws.H;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  const uint16_t* xr = x + (size_t)t * H;
  int shift = 0;
  if (mode == 0) {
    float m = 0.0f;
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(xr);
    for (int i = tid; i < H / 2; i += 256) {
      const uint32_t v = xw[i];
      m = fmaxf(m, fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    shift = token_shift(m);
  }
  for (int b = tid; b < H / 16; b += 256) prep_block(xr, b, t, ws, mode, xS, x_inv6S, shift);
  if (tid == 0) ws.xfac[t] = mode == 0 ? pow2f(shift) : xS;
}

// ------------------------------------------------------------------ quantiser hook
__global__ void __launch_bounds__(256) k_quantize_rows(const uint16_t* __restrict__ x, int rows,
                                                       int cols, float S, float inv6S,
                                                       uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_launch_dependents();
  const long long nblk = (long long)rows * (cols / 16);
  for (long long it = (long long)blockIdx.x * 256 + threadIdx.x; it < nblk;
       it += (long long)gridDim.x * 256) {
    const long long r = it / (cols / 16), b = it % (cols / 16);
    const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + b * 16);
    const uint4 u0 = src[0], u1 = src[1];
    const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(words[i]);
      v[2 * i + 1] = bf16_hi(words[i]);
    }
    uint32_t c[2];
    const uint32_t sf = quantize16(v, S, inv6S, c);
    *reinterpret_cast<uint2*>(codes + r * (cols / 2) + b * 8) = make_uint2(c[0], c[1]);
    scales[r * (cols / 16) + b] = static_cast<uint8_t>(sf);
  }
}


}  // namespace

size_t route_narrow_smem_bytes(int T, int H, int E, int k) {
  const size_t xbytes = (size_t)T * H * 2 + (size_t)kRouteRows * H * 2;
  const size_t fin = (size_t)T * k * 12 + (size_t)(E + 1) * 12 + 64;
  return xbytes > fin ? xbytes : fin;
}

cudaError_t launch_route_narrow(const LaunchCfg& lc, const uint16_t* x, const uint16_t* wr,
                                const WsView& ws, const PackView* pk, int mode, float xS,
                                float x_inv6S, int32_t* out_idx, float* out_w, int32_t* out_counts,
                                int32_t* out_offsets, int32_t* out_perm) {
  const PackView pkv = pk ? *pk : PackView{};
  const size_t smem = route_narrow_smem_bytes(ws.T, ws.H, ws.E, ws.k);
  RouteOut out{out_idx, out_w, out_counts, out_offsets, out_perm};
  const int grid = (ws.E + kRouteRows - 1) / kRouteRows;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(lc, kern, dim3(grid), dim3(256), smem, x, wr, ws, pkv, pk ? 1 : 0, mode, xS,
                  x_inv6S, out);
  };
  switch (ws.T) {
    case 1: return go(k_route_narrow<1>);
    case 2: return go(k_route_narrow<2>);
    case 3: return go(k_route_narrow<3>);
    case 4: return go(k_route_narrow<4>);
    case 5: return go(k_route_narrow<5>);
    case 6: return go(k_route_narrow<6>);
    case 7: return go(k_route_narrow<7>);
    default: return go(k_route_narrow<8>);
  }
}

cudaError_t launch_route_wide(const LaunchCfg& lc, const uint16_t* x, const uint16_t* wr,
                              const WsView& ws, const PackView* pk, int32_t* out_idx, float* out_w,
                              int32_t* out_counts, int32_t* out_offsets, int32_t* out_perm,
                              int* launches) {
  const PackView pkv = pk ? *pk : PackView{};
  RouteOut out{out_idx, out_w, out_counts, out_offsets, out_perm};
  cudaError_t e;
  const bool tc = ws.H % 64 == 0 && ((reinterpret_cast<uintptr_t>(x) |
                                       reinterpret_cast<uintptr_t>(wr)) & 15) == 0 &&
                  tc_supported();
  if (tc) {
    e = launch_tc_router(lc, x, wr, ws);
  } else {
    dim3 gg((ws.E + kGN - 1) / kGN, (ws.T + kGM - 1) / kGM);
    e = launch_kernel(lc, k_router_gemm, gg, dim3(256), 0, x, wr, ws);
  }
  if (e != cudaSuccess) return e;
  const int nchunk = (ws.T + kChunkTok - 1) / kChunkTok;
  e = launch_kernel(lc, k_topk_wide, dim3(nchunk), dim3(32 * kChunkTok), (size_t)ws.E * 8, ws, out);
  if (e != cudaSuccess) return e;
  e = launch_kernel(lc, k_scan_wide, dim3((ws.E + 31) / 32), dim3(1024), 0, ws, pkv, pk ? 1 : 0,
                    out, nchunk);
  if (e != cudaSuccess) return e;
  e = launch_kernel(lc, k_scatter_wide, dim3((ws.T * ws.k + 255) / 256), dim3(256), 0, ws, out);
  if (launches) *launches += 4;
  return e;
}

cudaError_t launch_xprep_wide(const LaunchCfg& lc, const uint16_t* x, const WsView& ws, int mode,
                              float xS, float x_inv6S) {
  return launch_kernel(lc, k_xprep_wide, dim3(ws.T), dim3(256), 0, x, ws, mode, xS, x_inv6S);
}

cudaError_t launch_quantize_rows(const LaunchCfg& lc, const uint16_t* x, int rows, int cols,
                                 float S, float inv6S, uint8_t* codes, uint8_t* scales) {
  const long long nblk = (long long)rows * (cols / 16);
  long long grid = (nblk + 255) / 256;
  const long long cap = (long long)lc.num_sms * 16;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_kernel(lc, k_quantize_rows, dim3((unsigned)grid), dim3(256), 0, x, rows, cols, S, inv6S,
                codes, scales);
}

}  // namespace moe
