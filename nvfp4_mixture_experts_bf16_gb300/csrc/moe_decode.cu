// moe_decode.cu — the whole routed-expert MoE step of a narrow call (T <= 8 tokens: decode and
// speculative verification) in ONE persistent kernel on sm_103a.
//
// The pages' engine runs this step as a chain of small kernels joined by programmatic dependent
// launch (release notes "Infernix windows-2026.10.11", section "Highlights"). At one token the
// step moves ~26 MB, about 4 us of HBM time, while every kernel boundary costs a few
// microseconds of drain, launch and first-copy latency, and every grid-wide barrier a couple of
// global round trips. Here one CTA per SM runs every phase, and CTAs never meet at a barrier:
// data that another CTA produces (logits, h, Y) is also written as 64-bit words {data, epoch of
// the call}, single-copy atomic, and the consumer polls the data itself (bounded) until it
// carries the current epoch. The epoch lives in the workspace; the last CTA of a call advances
// it.
//
//   1. router: each CTA copies its 3-4 router rows (TMA bulk copy, issued before waiting for
//      the preceding kernel: the router does not depend on it) and the T activation rows, and
//      writes its tagged logits (CUDA-core dot products for one or two tokens, mma.sync for
//      more). Then it converts the activations into the f16 (W4A16) or NVFP4-decoded (W4A4) MMA
//      operand in its own shared memory and writes its share of the W4A4 codes; with one or two
//      tokens the selecting warps skip that and route meanwhile.
//   2. routing: every CTA selects the top-k of every token itself (one warp per token, from the
//      tagged logits, by a threshold over the lane maxima), sorts the T*k selections by expert
//      and builds the expert groups in shared memory (one token: in the selecting warp, which
//      also issues the CTA's first gate/up copies). CTA 0 publishes idx / w / counts / offsets /
//      perm / slot_of after its own work. With a BF16 shared expert and one or two tokens (the
//      SH instantiations) the warps that do not select compute it meanwhile: h and its gate from
//      this CTA's gate/up rows (copied before the wait on the preceding kernel), exchanged as
//      tagged words, then this CTA's rows of its output Ys, tagged for the combine.
//   3. gate/up + SiLU*up: tasks (group, 16-row tile of I), as in the multi-kernel path; h is
//      written plain and tagged. As soon as its last gate/up stage is free, the producer warp
//      streams this CTA's down weights into the same shared memory.
//   4. down: tasks (group, 128-row tile of H); a task waits only for its own group's tagged h.
//      Each task writes Y (BF16) as pairs of rows, plain and tagged.
//   5. combine: 128-row tile j of out is formed, once its tagged Y has arrived, by the j-th CTA
//      in the order (late down tasks, CTA index), i.e. by CTAs done with their own down tasks
//      first: the fixed-order weighted sum over each token's k experts (rank order, FP32, then
//      BF16), plus sigma_t * BF16(Ys) of a shared expert. A layer of a chained stack
//      (moe_forward_layers) also writes the residual sum BF16(x + out), the next layer's input.
#include "moe_internal.cuh"
#include <type_traits>

namespace moe {
namespace {

constexpr int kDcWarps = 8;                       // consumer warps
constexpr int kDcThreads = (kDcWarps + 1) * 32;   // + one producer warp
constexpr int kDcCons = kDcWarps * 32;
constexpr int kDnRows = 128;                      // rows of H per down task (16 per warp)
constexpr int kDcSmemMax = 232448;                // 227 KB opt-in per block
constexpr int kDcStatic = 1024;                   // static shared memory allowance
constexpr int kShBatchIdx = 3;                    // shared expert: gate/up indices per batch
constexpr int kShBatchRows = 2 * kShBatchIdx;     //   (a gate row and an up row each)
constexpr int kShDnRows = 4;                      // shared expert: down rows per warp batch

// Prefetch of bytes (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// One expert's token group (<= 8 tokens) of the current call.
struct DcGroup {
  int expert, slot0, n;
  uint32_t toks;          // token of column c in bits 4c .. 4c+3
};
static_assert(sizeof(DcGroup) == 16, "DcGroup layout");

struct DcGeom {
  uint64_t wait_ns;             // bound of every wait (kWaitLimitNs unless a test shortens it)
  int skip_logits_cta;          // test fault injection: this CTA publishes no logits (-1: none)
  int rows_max;                 // router rows of one CTA, at most
  int rs;                       // bytes per staged router / activation row: 2H + 16 (padded so
                                // that 8 rows' fragment loads hit distinct banks)
  int KC, nkc, row_bytes;       // gate/up stage: KC reduction columns, nkc stages per task
  int gu_stage, gu_stages;
  int dn_stage, dn_stages;
  int arena;                    // router rows + raw x | gate/up ring | down ring
                                // | combine staging
  int x_stride;                 // 2H + 64: one x operand row
  int h_stride;                 // 2I + 16: one h operand row
  int xop;                      // x operand rows, later the h operand rows of one group
  int xsep;                     // one token: bytes of its own activation staging row (outside
                                // the arena, so the first weight copies can start early)
  int redbufs;                  // gate/up K-partial buffers: 2 when that still leaves two
                                // gate/up stages, else 1 (and a barrier after each epilogue)
  int smax, gmax;               // slots T*k, groups min(T*k, E)
  int smem;
  int sh_off;                   // shared expert inside the kernel: arena offsets of its gate/up
  int sh_hs;                    // rows and of its staged h
};

// Tagged words: {data in the low 32 bits, epoch of the writing call in the high 32 bits}, stored
// and loaded as single 64-bit accesses, which are single-copy atomic: a reader that sees the
// current epoch sees the data written with it, with no fence or barrier on either side.
__device__ __forceinline__ void st_tag(unsigned long long* p, uint32_t data, uint32_t ep) {
  const unsigned long long v = ((unsigned long long)ep << 32) | data;
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_tag(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t tag_of(unsigned long long v) { return (uint32_t)(v >> 32); }
__device__ __forceinline__ uint32_t data_of(unsigned long long v) { return (uint32_t)v; }

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ticket_acq_rel(uint32_t* ctr) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(ctr), "r"(1u)
               : "memory");
  return old;
}

// Top-k + softmax of one token from its tagged logits: polls (bounded) until every logit of
// the current epoch has arrived. False on timeout.
template <int V>
__device__ __forceinline__ bool topk_tagged_v(const unsigned long long* row, int E, int k,
                                              int lane, uint32_t ep, int& e_out, float& w_out,
                                              unsigned long long* cand, uint64_t limit_ns) {
  uint32_t key[V];
  uint32_t pending = 0;
  unsigned long long w[V];
#pragma unroll
  for (int i = 0; i < V; ++i)   // every load in flight before any is examined
    w[i] = lane + 32 * i < E ? ld_tag(row + lane + 32 * i) : 0ull;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    key[i] = 0u;
    if (lane + 32 * i < E) {
      if (tag_of(w[i]) == ep) key[i] = logit_key(__uint_as_float(data_of(w[i])));
      else pending |= 1u << i;
    }
  }
  bool ok = true;
  if (__any_sync(0xFFFFFFFFu, pending != 0u)) {
    const uint64_t t0 = globaltimer_ns();
    while (__any_sync(0xFFFFFFFFu, pending != 0u)) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if (pending & (1u << i)) {
          const unsigned long long w = ld_tag(row + lane + 32 * i);
          if (tag_of(w) == ep) {
            key[i] = logit_key(__uint_as_float(data_of(w)));
            pending &= ~(1u << i);
          }
        }
      }
      if (__any_sync(0xFFFFFFFFu, globaltimer_ns() - t0 > limit_ns)) {   // warp-uniform
        ok = false;
        break;
      }
    }
  }
  warp_select_scratch<V>(key, k, lane, cand, e_out, w_out);
  return ok;
}

__device__ __forceinline__ bool topk_tagged(const unsigned long long* row, int E, int k, int lane,
                                            uint32_t ep, int& e_out, float& w_out,
                                            unsigned long long* cand, uint64_t limit_ns) {
  // two register widths only: every instantiation is code that each CTA fetches once per launch
  if (E <= 512) return topk_tagged_v<16>(row, E, k, lane, ep, e_out, w_out, cand, limit_ns);
  return topk_tagged_v<32>(row, E, k, lane, ep, e_out, w_out, cand, limit_ns);
}

// Polls n tagged words (bounded) until all carry epoch ep. False on timeout.
template <int n>
__device__ __forceinline__ bool poll_tags(const unsigned long long* p, uint32_t ep,
                                          unsigned long long (&out)[n], uint64_t limit_ns) {
  bool all = true;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    out[i] = ld_tag(p + i);
    all &= tag_of(out[i]) == ep;
  }
  if (all) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    all = true;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      if (tag_of(out[i]) != ep) out[i] = ld_tag(p + i);
      all &= tag_of(out[i]) == ep;
    }
    if (all) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2,
                                               uint32_t b0, uint32_t b1) {
  // rows 8..15 of A are zero (a router CTA has at most 8 rows)
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// max(a, |b|) per BF16 lane of two packed pairs (a holds magnitudes)
__device__ __forceinline__ uint32_t bmax2_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b & 0x7FFF7FFFu));
  return d;
}

__device__ __forceinline__ int group_tok(uint32_t toks, int c) { return (toks >> (4 * c)) & 0xF; }

// Work split of a call. Gate/up tasks in contiguous ranges, the CTAs with one task fewer first
// (b < ns take R tasks, the others R + 1), so the first groups are computed entirely by CTAs
// that finish early. Up to one down task per such CTA, from those groups, is done early by
// them (while the other CTAs run their extra gate/up task); every other down task is spread
// over all CTAs (balanced), after the CTA's early one.
struct DcSplit {
  int q0, q1;     // gate/up tasks
  int de0, de1;   // early down tasks
  int dl0, dl1;   // late down tasks
  int crank;      // rank in the order (late down tasks, b): the combine's tile order, so that
                  // the CTAs that finish their down tasks first form the output tiles
};
__device__ __forceinline__ DcSplit dc_split(int U, int gu_tiles, int dn_tiles) {
  const int G = gridDim.x, b = blockIdx.x;
  const int NG = U * gu_tiles, ND = U * dn_tiles;
  const int R = NG / G, Rx = NG % G, ns = G - Rx;
  DcSplit sp;
  sp.q0 = b < ns ? b * R : ns * R + (b - ns) * (R + 1);
  sp.q1 = sp.q0 + (b < ns ? R : R + 1);
  const int eg = Rx > 0 ? (ns * R) / gu_tiles : 0;   // groups whose tasks all lie on b < ns
  const int NE = min(eg * dn_tiles, ns), NL = ND - NE;
  sp.de0 = sp.de1 = 0;
  if (b < ns && NE > 0) {
    sp.de0 = (int)((long long)NE * b / ns);
    sp.de1 = (int)((long long)NE * (b + 1) / ns);
  }
  sp.dl0 = NE + (int)((long long)NL * b / G);
  sp.dl1 = NE + (int)((long long)NL * (b + 1) / G);
  // L = NL / G late tasks for most CTAs, L + 1 for NL % G of them; among the CTAs before b,
  // (dl0 - NE) - L * b have L + 1
  const int L = NL / G, nlow = G - NL % G, hi_before = (sp.dl0 - NE) - L * b;
  sp.crank = (sp.dl1 - sp.dl0 == L) ? b - hi_before : nlow + hi_before;
  return sp;
}

template <int NT, int MODE, bool SH>
__global__ void __launch_bounds__(kDcThreads, 1)
    k_decode(PackView pk, WsView ws, DcGeom geo, const uint16_t* __restrict__ x,
             const uint16_t* __restrict__ wr, float xS, float x_inv6S,
             uint16_t* __restrict__ out, uint16_t* __restrict__ xnext, int a8, ShView sv) {
  // SH: the shared expert runs inside this launch (one or two tokens)
  static_assert(!SH || NT <= 2, "the shared expert is fused for one or two tokens");
  // 0: W4A16, 1: quantised activations (one instantiation each: smaller code): NVFP4 (W4A4), or
  // E4M3 (W4A8) when a8 is set; both run the same f16 MMAs on exactly decoded values
  constexpr int mode = MODE;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* arena = smem;
  unsigned char* xop = arena + geo.arena;
  // [redbufs][8 warps][2][128]: with two buffers gate/up task q's K-partials go to buffer
  // q % 2, so the next task's warps need not wait for this task's epilogue
  float* red = reinterpret_cast<float*>(xop + geo.xop);
  DcGroup* grp = reinterpret_cast<DcGroup*>(red + geo.redbufs * kDcWarps * 2 * 128);
  int32_t* sel_idx = reinterpret_cast<int32_t*>(grp + geo.gmax);        // [S]
  float* sel_w = reinterpret_cast<float*>(sel_idx + geo.smax);          // [S]
  int32_t* sel_slot = reinterpret_cast<int32_t*>(sel_w + geo.smax);     // [S]
  // the selections sorted by expert (own region: the arena only ever receives TMA writes and
  // the combine's staging, so no proxy fence is needed before the first weight copy)
  int32_t* sorted_e = sel_slot + geo.smax;                               // [S] expert of slot p
  int32_t* sorted_t = sorted_e + geo.smax;                               // [S] token of slot p
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(sorted_t + geo.smax) + 7) & ~uintptr_t(7));
  uint64_t* gfull = bars;
  uint64_t* gempty = gfull + geo.gu_stages;
  uint64_t* dfull = gempty + geo.gu_stages;
  uint64_t* dempty = dfull + geo.dn_stages;
  uint64_t* rbar = dempty + geo.dn_stages;
  uint64_t* xbar = rbar + 1;
  uint64_t* sbar = xbar + 1;   // the shared expert's gate/up rows (SH)
  unsigned char* xsep_row = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sbar + 1) + 15) & ~uintptr_t(15));
  __shared__ float xfac_s[NT];
  __shared__ int shift_s[NT];
  __shared__ float hfac_s[kGroup];
  __shared__ uint32_t hamax_s[kGroup];
  __shared__ int wcount_s[kDcWarps + 1];
  __shared__ volatile int abort_s;
  // shared expert (SH): per-warp partial sums of one batch of its gate/up rows
  __shared__ float shp_s[SH ? (kDcWarps + 1) * kShBatchRows * NT : 1];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int T = NT;
  const int H = ws.H, E = ws.E, k = ws.k, I = ws.I, S = T * k;
  const int G = gridDim.x, b = blockIdx.x;
  const int row0 = (E * b) / G;
  const int nrows = (E * (b + 1)) / G - row0;
  unsigned char* wrs = arena;                                            // [rows][rs bytes]
  unsigned char* xraw = geo.xsep ? xsep_row                              // [T][rs bytes]
                                 : arena + (size_t)geo.rows_max * geo.rs;

  if (tid == 0) {
    for (int s = 0; s < geo.gu_stages; ++s) {
      mbar_init(&gfull[s], 1);
      mbar_init(&gempty[s], kDcWarps);
    }
    for (int s = 0; s < geo.dn_stages; ++s) {
      mbar_init(&dfull[s], 1);
      mbar_init(&dempty[s], kDcWarps);
    }
    mbar_init(rbar, 1);
    mbar_init(xbar, 1);
    mbar_init(sbar, 1);
    fence_mbar_init();
    abort_s = 0;
    // the router rows are weights: copy them before waiting for the preceding kernel
    if (nrows > 0) {
      mbar_arrive_expect_tx(rbar, (uint32_t)nrows * H * 2);
      for (int r = 0; r < nrows; ++r)
        bulk_g2s(wrs + (size_t)r * geo.rs, wr + (size_t)(row0 + r) * H, (uint32_t)H * 2, rbar);
    }
    if constexpr (SH) {
      // the shared expert's weights: this CTA's gate/up rows (indices [j0, j1) of 0..Is, index
      // Is being the gate vector) into the arena past the first gate/up stage, and its down
      // rows [r0, r1) of H towards L2 (read once its h is complete)
      const int Is = sv.Is;
      const int j0 = (int)((long long)(Is + 1) * b / G), j1 = (int)((long long)(Is + 1) * (b + 1) / G);
      uint32_t bytes = 0;
      for (int j = j0; j < j1; ++j) bytes += (j < Is ? 2u : 1u) * (uint32_t)H * 2;
      if (bytes > 0) {
        mbar_arrive_expect_tx(sbar, bytes);
        unsigned char* dst = arena + geo.sh_off;
        for (int j = j0; j < j1; ++j) {
          const int jj = j - j0;
          if (j < Is) {
            bulk_g2s(dst + (size_t)(2 * jj) * H * 2, sv.gate_up + (size_t)j * H, (uint32_t)H * 2, sbar);
            bulk_g2s(dst + (size_t)(2 * jj + 1) * H * 2, sv.gate_up + (size_t)(Is + j) * H,
                     (uint32_t)H * 2, sbar);
          } else {
            bulk_g2s(dst + (size_t)(2 * jj) * H * 2, sv.gate, (uint32_t)H * 2, sbar);
          }
        }
      }
      const int r0 = (int)((long long)H * b / G), r1 = (int)((long long)H * (b + 1) / G);
      if (r1 > r0) l2_prefetch(sv.down + (size_t)r0 * Is, (uint32_t)(r1 - r0) * Is * 2);
    }
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) {
    mbar_arrive_expect_tx(xbar, (uint32_t)T * H * 2);
    for (int t = 0; t < T; ++t)
      bulk_g2s(xraw + (size_t)t * geo.rs, x + (size_t)t * H, (uint32_t)H * 2, xbar);
  }
  // this call's epoch: one past the last completed call's (never 0, the zeroed workspace's tag)
  uint32_t ep = __ldcg(&ws.ctl[kCtlEpoch]) + 1u;
  if (ep == 0u) ep = 1u;
  if ((nrows > 0 && !mbar_wait(rbar, 0, geo.wait_ns)) || !mbar_wait(xbar, 0, geo.wait_ns)) {
    record_status(ws.ctl, kStTimeout);
    abort_s = 1;
  }

  // ---------------- 1. router rows on the tensor cores: logits[t][row0 + r] = W[r] . x[t] as one
  // m16n8k16 BF16 MMA chain per warp over an eighth of H (A = the CTA's <= 8 router rows,
  // B = the T tokens, FP32 accumulation; the products are exact). The B fragments also give each
  // token's max |x| (for the f16 operand's scaling).
  float* amax_part = red + kDcWarps * 64;   // [8 warps][8 tokens]
  if (NT <= 2 && warp < kDcWarps) {
    // one or two tokens: FP32 dot products on the CUDA cores (an MMA chain would leave 7 of
    // its 8 columns empty): lane l of warp w takes the 8-element chunks 32 (2w + h) + l,
    // h = 0, 1 (and every 512 chunks further), so that a warp's loads are 512 contiguous bytes
    // (exact BF16 products, FP32 sums), then a butterfly over the warp. Also each token's
    // max |x| over the thread's chunks.
    float am[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) am[t] = 0.0f;
    // rows in groups of 4 (the CTA holds 3-4 rows at 512 experts): no work is issued for
    // absent rows beyond the group; one pass at least, for the max |x| (a CTA may hold no row)
    for (int r0 = 0; r0 < (nrows > 0 ? nrows : 1); r0 += 4) {
      float acc[4][NT];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = 0.0f;
      for (int c8 = warp * 64 + lane; c8 < H / 8; c8 += kDcCons * 2) {
        const int o0 = c8 * 16, o1 = (c8 + 32) * 16;   // byte offsets of the two chunks
        const bool h1 = c8 + 32 < H / 8;                  // H % 512 != 0: a last half chunk
        float xv[NT][16];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 u0 = lds128(xraw + (size_t)t * geo.rs + o0);
          const uint4 u1 = h1 ? lds128(xraw + (size_t)t * geo.rs + o1) : make_uint4(0, 0, 0, 0);
          const uint32_t wd[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          uint32_t m2 = 0u;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            xv[t][2 * i] = bf16_lo(wd[i]);
            xv[t][2 * i + 1] = bf16_hi(wd[i]);
            m2 = bmax2_abs(m2, wd[i]);
          }
          am[t] = fmaxf(am[t], fmaxf(bf16_lo(m2), bf16_hi(m2)));
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (r0 + r < nrows) {
            const unsigned char* wrow = wrs + (size_t)(r0 + r) * geo.rs;
            const uint4 u0 = lds128(wrow + o0);
            const uint4 u1 = h1 ? lds128(wrow + o1) : make_uint4(0, 0, 0, 0);
            const uint32_t wd[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float w0 = bf16_lo(wd[i]), w1 = bf16_hi(wd[i]);
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                acc[r][t] = fmaf(w0, xv[t][2 * i], acc[r][t]);
                acc[r][t] = fmaf(w1, xv[t][2 * i + 1], acc[r][t]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if (r0 + r < nrows) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            float v = acc[r][t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0) red[(warp * 8 + r0 + r) * 8 + t] = v;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float m = am[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
      if (lane == 0) amax_part[warp * 8 + t] = m;
    }
  } else if (warp < kDcWarps) {
    const int g = lane >> 2, c = lane & 3;
    const bool arow = g < nrows, bcol = g < T;
    const int kw = H / kDcWarps;                       // K range of this warp
    const unsigned char* ap = wrs + (size_t)g * geo.rs + (size_t)(warp * kw + 2 * c) * 2;
    const unsigned char* bp = xraw + (size_t)g * geo.rs + (size_t)(warp * kw + 2 * c) * 2;
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t am2 = 0u;   // running max |x| of the B fragments, two BF16 lanes
#pragma unroll 2
    for (int ks = 0; ks < kw / 16; ks += 2) {
      uint32_t a[4] = {0u, 0u, 0u, 0u}, bb[4] = {0u, 0u, 0u, 0u};
      if (arow) {
        a[0] = lds32(ap + ks * 32);
        a[1] = lds32(ap + ks * 32 + 16);
        a[2] = lds32(ap + ks * 32 + 32);
        a[3] = lds32(ap + ks * 32 + 48);
      }
      if (bcol) {
        bb[0] = lds32(bp + ks * 32);
        bb[1] = lds32(bp + ks * 32 + 16);
        bb[2] = lds32(bp + ks * 32 + 32);
        bb[3] = lds32(bp + ks * 32 + 48);
      }
      mma_bf16_16816(d0, a[0], a[1], bb[0], bb[1]);
      mma_bf16_16816(d1, a[2], a[3], bb[2], bb[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) am2 = bmax2_abs(am2, bb[q]);
    }
    float am = fmaxf(bf16_lo(am2), bf16_hi(am2));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    // D[row g][token 2c, 2c+1]
    red[(warp * 8 + g) * 8 + 2 * c] = d0[0] + d1[0];
    red[(warp * 8 + g) * 8 + 2 * c + 1] = d0[1] + d1[1];
    if (c == 0) amax_part[warp * 8 + g] = am;
  }
  __syncthreads();
  if (tid < nrows * T && b != geo.skip_logits_cta) {
    const int rl = tid / T, t = tid % T;
    float s = red[rl * 8 + t];
#pragma unroll
    for (int w = 1; w < kDcWarps; ++w) s += red[(w * 8 + rl) * 8 + t];
    unsigned long long* lg = reinterpret_cast<unsigned long long*>(ws.logits);
#pragma unroll
    for (int rep = 0; rep < kLogitReplicas; ++rep)
      st_tag(lg + ((size_t)rep * T + t) * E + row0 + rl, __float_as_uint(s), ep);
  } else if (tid >= kDcCons && tid - kDcCons < T) {
    const int t = tid - kDcCons;
    float m = amax_part[t];
#pragma unroll
    for (int w = 1; w < kDcWarps; ++w) m = fmaxf(m, amax_part[w * 8 + t]);
    shift_s[t] = token_shift(m);
    xfac_s[t] = mode == 0 ? pow2f(shift_s[t]) : (a8 ? __fmul_rn(6.0f, xS) : xS);
  }
  __syncthreads();
  if (warp == kDcWarps) {
    if (mode != 0) {
      // W4A4 / W4A8: this CTA's share of the quantised activations (16-element blocks b,
      // b + G, ...), written plain while the consumer warps wait for the logits. Every CTA's
      // operand build (2b) decodes all T tokens from them instead of quantising them itself.
      const int nb = H / 16;
      for (int blk = b + G * lane; blk < T * nb; blk += G * 32) {
        const int t = blk / nb, bb = blk % nb;
        const uint4* src = reinterpret_cast<const uint4*>(xraw + (size_t)t * geo.rs + bb * 32);
        const uint4 u0 = src[0], u1 = src[1];
        const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = bf16_lo(words[i]);
          v[2 * i + 1] = bf16_hi(words[i]);
        }
        if (a8) {
          uint32_t cw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int i = 0; i < 16; ++i) cw[i >> 2] |= a8_encode(v[i], x_inv6S) << (8 * (i & 3));
          *reinterpret_cast<uint4*>(ws.xq + (size_t)t * H + bb * 16) =
              make_uint4(cw[0], cw[1], cw[2], cw[3]);
        } else {
          uint32_t codes[2];
          const uint32_t sf = quantize16(v, xS, x_inv6S, codes);
          *reinterpret_cast<uint2*>(ws.xq + (size_t)t * (H / 2) + bb * 8) =
              make_uint2(codes[0], codes[1]);
          ws.xsf[(size_t)t * (H / 16) + bb] = static_cast<uint8_t>(sf);
        }
      }
    }
    // every launch counts its CTAs here (all modes), so the counter stays at (epoch - 1) * G
    // at the start of a call on this workspace; the release orders the warp's share before it
    __syncwarp();
    if (lane == 0) (void)ticket_acq_rel(&ws.ctl[kCtlXShare]);
  }

  // ---------------- 2a. top-k + softmax of every token (warp t), from the tagged logits. With
  // T <= 2 the selection runs while the other warps build the activation operand (below);
  // with more tokens every warp takes part in the operand first.
  constexpr bool kEarlyTopk = NT <= 2;
  const int gu_tiles = I / 16, dn_tiles = H / kDnRows;
  // this CTA's gate/up tasks [q0, q1) (one token: U = k groups, known before the routing)
  int q0 = 0, q1 = 0;
  if (T == 1) {
    const DcSplit sp1 = dc_split(k, gu_tiles, H / kDnRows);
    q0 = sp1.q0;
    q1 = sp1.q1;
  }
  // one token: the selecting warp issues the first gate/up stages itself, right after the
  // selection (the arena holds no staged activations then, and every router row is consumed)
  // (the first stage only: the CTA's later stages follow once it has landed, so that every
  // CTA's first stage gets the memory system before anyone's second)
  const int npre = (T == 1 && geo.xsep && q1 > q0) ? 1 : 0;

  // copies of gate/up stage `chunk` = (task q, k-chunk kc) of expert e into its ring slot
  auto issue_gu = [&](int chunk, int q, int kc, int e) {
    const int it = q % gu_tiles, s = chunk % geo.gu_stages;
    const uint32_t half = geo.row_bytes;
    const size_t grow0 = (size_t)e * I + (size_t)it * 16;
    const uint8_t* gsrc = pk.gate_codes + grow0 * (H / 2);
    const uint8_t* usrc = pk.up_codes + grow0 * (H / 2);
    const uint8_t* gsc = pk.gu_scales + (((size_t)0 * pk.E + e) * gu_tiles + it) * (size_t)H;
    const uint8_t* usc = pk.gu_scales + (((size_t)1 * pk.E + e) * gu_tiles + it) * (size_t)H;
    unsigned char* st = arena + (size_t)s * geo.gu_stage;
    mbar_arrive_expect_tx(&gfull[s], 32 * half + 2 * geo.KC);
    if (geo.nkc == 1) {
      bulk_g2s(st, gsrc, 16 * half, &gfull[s]);
      bulk_g2s(st + 16 * half, usrc, 16 * half, &gfull[s]);
    } else {
      for (int r = 0; r < 16; ++r) {
        bulk_g2s(st + r * half, gsrc + (size_t)r * (H / 2) + (size_t)kc * half, half, &gfull[s]);
        bulk_g2s(st + (16 + r) * half, usrc + (size_t)r * (H / 2) + (size_t)kc * half, half,
                 &gfull[s]);
      }
    }
    bulk_g2s(st + 32 * half, gsc + (size_t)kc * geo.KC, geo.KC, &gfull[s]);
    bulk_g2s(st + 32 * half + geo.KC, usc + (size_t)kc * geo.KC, geo.KC, &gfull[s]);
  };

  auto select_token = [&]() {
    int e_sel;
    float w_sel;
    const unsigned long long* lg = reinterpret_cast<const unsigned long long*>(ws.logits) +
                                   ((size_t)(b % kLogitReplicas) * T + warp) * E;
    // scratch: 32 words per warp in the GEMV partials buffer (free once the logits are out)
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(red) + warp * 32;
    const bool ok = topk_tagged(lg, E, k, lane, ep, e_sel, w_sel, cand, geo.wait_ns);
    if (!ok && lane == 0) {
      record_status(ws.ctl, kStTimeout);
      abort_s = 1;
    }
    if (T == 1) {
      // one token: its k experts are distinct, so every selection is a group of one, and
      // the slot of selection j is its rank by expert (k shuffles, no block barrier)
      int p = 0;
#pragma unroll 4
      for (int j = 0; j < k; ++j) p += __shfl_sync(0xFFFFFFFFu, e_sel, j) < e_sel;
      if (lane < k) {
        sel_idx[lane] = e_sel;
        sel_w[lane] = w_sel;
        sel_slot[lane] = p;
        sorted_e[p] = e_sel;
        sorted_t[p] = 0;
        DcGroup gr;
        gr.expert = e_sel;
        gr.slot0 = p;
        gr.n = 1;
        gr.toks = 0u;
        grp[p] = gr;
      }
      if (__all_sync(0xFFFFFFFFu, ok && !abort_s)) {
        for (int c = 0; c < npre; ++c) {
          const int q = q0 + c / geo.nkc;
          const unsigned src = __ballot_sync(0xFFFFFFFFu, lane < k && p == q / gu_tiles);
          const int e = __shfl_sync(0xFFFFFFFFu, e_sel, __ffs(src) - 1);
          if (lane == c) issue_gu(c, q, c % geo.nkc, e);
        }
      }
    } else if (lane < k) {
      sel_idx[warp * k + lane] = e_sel;
      sel_w[warp * k + lane] = w_sel;
    }
  };
  // the quantised modes select before building the operand: the operand's codes come from the
  // other CTAs' tagged words, published while the logits are exchanged, and the selection's
  // time lets them land before anyone polls (every thread polling early floods L2 with spinning
  // loads and delays the very stores it waits for)
  constexpr bool kSelectFirst = kEarlyTopk || MODE != 0;
  if (kSelectFirst && warp < T) select_token();

  // ---------------- shared expert (SH: one or two tokens), while warps 0 .. T-1 select. The
  // other warps form g = Wg[j] . x_t and u = Wu[j] . x_t for this CTA's indices j (FP32 sums of
  // exact BF16 products), then hs = BF16(SiLU(g) * u), or sigma_t = 1 / (1 + exp(-gv . x_t)) for
  // the gate vector, written plain and tagged; then, once every CTA's hs words have arrived,
  // Ys[t][r] = Wd[r] . hs_t for this CTA's rows [r0, r1) of H (their weights loaded into
  // registers before the wait), written plain (FP32) and tagged for the combine. The gate/up
  // rows and the staged hs sit in the arena past the first gate/up stage, which no copy reaches
  // before the barrier after the operand build (2b); one token's consumers wait on its first
  // gate/up stage after that barrier anyway, so this work stays off the critical path.
  if constexpr (SH) {
    if (warp >= T) {
      const int Is = sv.Is, nthr = (kDcWarps + 1 - T) * 32, i0 = tid - 32 * T;
      const int j0 = (int)((long long)(Is + 1) * b / G), j1 = (int)((long long)(Is + 1) * (b + 1) / G);
      const unsigned char* rows = arena + geo.sh_off;
      const int nunits = H / 8;
      unsigned long long* htag = ws.sh_tag;
      unsigned long long* stag = htag + (size_t)T * Is;
      unsigned long long* ytag = stag + T;
      if (j1 > j0 && !mbar_wait(sbar, 0, geo.wait_ns)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      for (int jb = j0; jb < j1; jb += kShBatchIdx) {
        float acc[kShBatchRows][NT];
#pragma unroll
        for (int r = 0; r < kShBatchRows; ++r)
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[r][t] = 0.0f;
        for (int u = i0; u < nunits; u += nthr) {
          uint4 xv[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) xv[t] = lds128(xraw + (size_t)t * geo.rs + u * 16);
#pragma unroll
          for (int r = 0; r < kShBatchRows; ++r) {
            const int j = jb + r / 2;
            if (j < j1 && (j < Is || (r & 1) == 0)) {
              const uint4 wv =
                  lds128(rows + (size_t)(2 * (j - j0) + (r & 1)) * H * 2 + (size_t)u * 16);
#pragma unroll
              for (int t = 0; t < NT; ++t) acc[r][t] += dot8_bf16(wv, xv[t]);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < kShBatchRows; ++r)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            float v = acc[r][t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0) shp_s[(warp * kShBatchRows + r) * NT + t] = v;
          }
        asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
        if (i0 < kShBatchIdx * NT) {
          const int q = i0 / NT, t = i0 % NT, j = jb + q;
          if (j < j1) {
            // the warps' partials in a fixed order
            float g = 0.0f, uu = 0.0f;
            for (int w = T; w <= kDcWarps; ++w) {
              g += shp_s[(w * kShBatchRows + 2 * q) * NT + t];
              uu += shp_s[(w * kShBatchRows + 2 * q + 1) * NT + t];
            }
            if (j < Is) {
              const uint16_t hb = f32_to_bf16_rn(silu_mul(g, uu));
              sv.hs[(size_t)t * Is + j] = hb;
              st_tag(htag + (size_t)t * Is + j, hb, ep);
            } else {
              const float sg = 1.0f / (1.0f + expf(-g));
              sv.sigma[t] = sg;
              st_tag(stag + t, __float_as_uint(sg), ep);
            }
          }
        }
        asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");   // shp_s is reused
      }
      // down: warp wi of nw takes rows r0 + wi + nw * i, lanes the 16-byte units of a row
      const int r0 = (int)((long long)H * b / G), r1 = (int)((long long)H * (b + 1) / G);
      const int nw = kDcWarps + 1 - T, wi = warp - T, nu = Is / 8;
      uint16_t* hsm = reinterpret_cast<uint16_t*>(arena + geo.sh_hs);
      uint4 wd[kShDnRows][2];
      auto load_rows = [&](int rb) {
#pragma unroll
        for (int rr = 0; rr < kShDnRows; ++rr) {
          const int r = r0 + wi + nw * (rb + rr);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int u = lane + 32 * c;
            wd[rr][c] = (r < r1 && u < nu)
                            ? __ldg(reinterpret_cast<const uint4*>(sv.down + (size_t)r * Is) + u)
                            : make_uint4(0u, 0u, 0u, 0u);
          }
        }
      };
      load_rows(0);
      for (int idx = i0; idx < T * Is; idx += nthr) {
        unsigned long long w[1];
        if (!poll_tags<1>(htag + idx, ep, w, geo.wait_ns)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        hsm[idx] = static_cast<uint16_t>(data_of(w[0]));
      }
      asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
      for (int rb = 0; r0 + wi + nw * rb < r1; rb += kShDnRows) {
        if (rb > 0) load_rows(rb);
        float acc[kShDnRows][NT];
#pragma unroll
        for (int rr = 0; rr < kShDnRows; ++rr)
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[rr][t] = 0.0f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int u = lane + 32 * c;
          if (u < nu) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const uint4 hv = lds128(reinterpret_cast<const unsigned char*>(hsm + (size_t)t * Is + u * 8));
#pragma unroll
              for (int rr = 0; rr < kShDnRows; ++rr) acc[rr][t] += dot8_bf16(wd[rr][c], hv);
            }
          }
        }
        // units past the register-held ones (Is > 512)
        for (int u = 64 + lane; u < nu; u += 32) {
#pragma unroll
          for (int rr = 0; rr < kShDnRows; ++rr) {
            const int r = r0 + wi + nw * (rb + rr);
            if (r < r1) {
              const uint4 wv = __ldg(reinterpret_cast<const uint4*>(sv.down + (size_t)r * Is) + u);
#pragma unroll
              for (int t = 0; t < NT; ++t)
                acc[rr][t] += dot8_bf16(wv, lds128(reinterpret_cast<const unsigned char*>(hsm + (size_t)t * Is + u * 8)));
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < kShDnRows; ++rr) {
          const int r = r0 + wi + nw * (rb + rr);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            float v = acc[rr][t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0 && r < r1) {
              sv.ys[(size_t)t * H + r] = v;
              st_tag(ytag + (size_t)t * H + r, __float_as_uint(v), ep);
            }
          }
        }
      }
    }
  }

  // ---------------- 2b. activation operand of every token, in this CTA's shared memory
  {
    const int nb = H / 16;
    const int t0 = kEarlyTopk ? 32 * T : 0;
    const int stride = kDcThreads - t0;
    // element 128J + 32c + 8p + q of a row is stored at 128J + 32p + 8c + q
    auto store_op = [&](int t, int bb, const uint32_t (&hw)[8]) {
      const int J = bb >> 3, c = (bb & 7) >> 1, p0 = 2 * (bb & 1);
      unsigned char* row = xop + (size_t)t * geo.x_stride + (size_t)(J * 128 + 8 * c) * 2;
      *reinterpret_cast<uint4*>(row + 64 * p0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(row + 64 * (p0 + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    };
    if (mode == 0) {
      for (int blk = tid - t0; blk < T * nb; blk += stride) {
        if (blk < 0) break;
        const int t = blk / nb, bb = blk % nb;
        const uint4* src = reinterpret_cast<const uint4*>(xraw + (size_t)t * geo.rs + bb * 32);
        const uint4 u0 = src[0], u1 = src[1];
        const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float f = pow2f(-shift_s[t]);
        uint32_t hw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const __half2 h2 = __halves2half2(__float2half_rn(__fmul_rn(bf16_lo(words[i]), f)),
                                            __float2half_rn(__fmul_rn(bf16_hi(words[i]), f)));
          hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        store_op(t, bb, hw);
      }
    } else {
      // W4A4 / W4A8: the codes every CTA published (its share above), read once all G CTAs
      // have counted theirs for this call; four consecutive blocks (one token) per item, all
      // of a thread's loads issued before any is used. The f16 operand is the code's value:
      // E2M1 x E4M3 scale has at most 6 significant bits and lies between 2^-10 and 2688 in
      // magnitude (exact in f16); E4M3 codes are exact in f16.
      if (tid == 0) {
        const uint32_t target = ep * (uint32_t)G;
        const uint64_t tw0 = globaltimer_ns();
        while ((int32_t)(ld_acquire_u32(&ws.ctl[kCtlXShare]) - target) < 0) {
          if (globaltimer_ns() - tw0 > geo.wait_ns) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
        }
      }
      __syncthreads();
      const int nitems = T * nb / 4;
      constexpr int kIt = 2;   // items per thread per round
      for (int base = tid; base < nitems; base += kIt * kDcThreads) {
        uint4 cv[kIt][4];
        uint32_t sfw[kIt];
#pragma unroll
        for (int u = 0; u < kIt; ++u) {
          const int it = base + u * kDcThreads;
          if (it >= nitems) break;
          const int t = it / (nb / 4), bb = (it % (nb / 4)) * 4;
          if (a8) {
            const uint4* c = reinterpret_cast<const uint4*>(ws.xq + (size_t)t * H + bb * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) cv[u][i] = __ldcg(c + i);
          } else {
            const uint4* c = reinterpret_cast<const uint4*>(ws.xq + (size_t)t * (H / 2) + bb * 8);
            cv[u][0] = __ldcg(c);
            cv[u][1] = __ldcg(c + 1);
            sfw[u] = __ldcg(reinterpret_cast<const uint32_t*>(ws.xsf + (size_t)t * (H / 16) + bb));
          }
        }
#pragma unroll
        for (int u = 0; u < kIt; ++u) {
          const int it = base + u * kDcThreads;
          if (it >= nitems) break;
          const int t = it / (nb / 4), bb = (it % (nb / 4)) * 4;
#pragma unroll
          for (int q = 0; q < 4; ++q) {   // block bb + q
            uint32_t hw[8];
            if (a8) {
              const uint32_t w4[4] = {cv[u][q].x, cv[u][q].y, cv[u][q].z, cv[u][q].w};
#pragma unroll
              for (int i = 0; i < 8; ++i) hw[i] = e4m3x2_to_f16x2(w4[i >> 1] >> (16 * (i & 1)));
            } else {
              const uint4 cc = cv[u][q >> 1];
              const uint32_t lo = (q & 1) ? cc.z : cc.x, hi = (q & 1) ? cc.w : cc.y;
              const uint32_t s2 = e4m3x2_to_f16x2((sfw[u] >> (8 * q)) & 0xFFu);
              uint32_t f[8];
              e2m1x8_to_f16x2x4(lo, *reinterpret_cast<uint32_t(*)[4]>(&f[0]));
              e2m1x8_to_f16x2x4(hi, *reinterpret_cast<uint32_t(*)[4]>(&f[4]));
#pragma unroll
              for (int i = 0; i < 8; ++i) hw[i] = hmul2_lo(f[i], s2);
            }
            store_op(t, bb + q, hw);
          }
        }
      }
    }
  }
  __syncthreads();
  if (!kSelectFirst && warp < T) select_token();

  // ---------------- 2c. groups, in every CTA: a stable sort of the S = T*k selections by
  // expert (entry s = t*k + j goes to slot #{s' : e_s' < e_s} + #{s' < s : e_s' == e_s}) and one
  // group per distinct expert, numbered in slot order. One token: done in the selecting warp.
  int U = 0;
  if (T == 1) {
    U = k;
  } else {
  if (!kEarlyTopk) __syncthreads();
  if (tid < S) {
    const int e = sel_idx[tid];
    int p = 0;
    for (int s2 = 0; s2 < S; ++s2) {
      const int e2 = sel_idx[s2];
      p += (e2 < e) || (e2 == e && s2 < tid);
    }
    sel_slot[tid] = p;
    sorted_e[p] = e;
    sorted_t[p] = tid / k;
  }
  __syncthreads();
  // one group per distinct expert (at most T <= 8 slots each), numbered in slot order
  const bool gstart = tid < S && (tid == 0 || sorted_e[tid] != sorted_e[tid - 1]);
  const unsigned gbal = __ballot_sync(0xFFFFFFFFu, gstart);
  if (lane == 0) wcount_s[warp] = __popc(gbal);
  __syncthreads();
  int ubase = 0;
#pragma unroll
  for (int w = 0; w <= kDcWarps; ++w) {
    if (w < warp) ubase += wcount_s[w];
    U += wcount_s[w];
  }
  if (gstart) {
    const int e = sorted_e[tid];
    int n = 1;
    while (tid + n < S && sorted_e[tid + n] == e) ++n;
    uint32_t toks = 0;
    for (int r = 0; r < n; ++r) toks |= (uint32_t)sorted_t[tid + r] << (4 * r);
    DcGroup gr;
    gr.expert = e;
    gr.slot0 = tid;
    gr.n = n;
    gr.toks = toks;
    grp[ubase + __popc(gbal & ((1u << lane) - 1u))] = gr;
  }
  __syncthreads();
  }
  // groups and selections are final from here on (one token: since the operand barrier)

  const DcSplit sp = dc_split(U, gu_tiles, dn_tiles);
  q0 = sp.q0;
  q1 = sp.q1;
  // this CTA's down tasks, early ones first: task i of nd is q = dq(i)
  const int nde = sp.de1 - sp.de0, nd = nde + (sp.dl1 - sp.dl0);
  auto dq = [&](int i) { return i < nde ? sp.de0 + i : sp.dl0 + (i - nde); };

  if (warp == kDcWarps) {
    // ---------------- producer: gate/up tasks, then this CTA's down tasks
    if (lane != 0) return;
    int chunk = 0;
    for (int q = q0; q < q1 && !abort_s; ++q) {
      const int e = grp[q / gu_tiles].expert;
      for (int kc = 0; kc < geo.nkc; ++kc, ++chunk) {
        if (chunk < npre) continue;   // issued by the selecting warp
        const int s = chunk % geo.gu_stages, n = chunk / geo.gu_stages;
        if (n > 0 && !mbar_wait(&gempty[s], (n - 1) & 1, geo.wait_ns)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
          break;
        }
        // one token: the second task's stage waits for the first to land (its only completed
        // phase)
        if (npre > 0 && chunk == 1 && geo.nkc == 1 && !mbar_wait(&gfull[0], 0, geo.wait_ns)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
          break;
        }
        issue_gu(chunk, q, kc, e);
      }
    }
    // the arena becomes the down ring once the consumers have released every gate/up stage
    const int used = chunk < geo.gu_stages ? chunk : geo.gu_stages;
    for (int i = 0; i < used; ++i) {
      // landed (after a timeout elsewhere the consumers may release a stage they did not read)
      // and released
      const int c2 = chunk - 1 - i;
      if (!mbar_wait(&gfull[c2 % geo.gu_stages], (c2 / geo.gu_stages) & 1, geo.wait_ns) ||
          !mbar_wait(&gempty[c2 % geo.gu_stages], (c2 / geo.gu_stages) & 1, geo.wait_ns)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
    }
    const uint32_t code_bytes = (uint32_t)kDnRows * (I / 2);
    int dchunk = 0;
    for (int i = 0; i < nd && !abort_s; ++i, ++dchunk) {
      const int q = dq(i);
      const int gi = q / dn_tiles, ht = q % dn_tiles;
      const int e = grp[gi].expert;
      const int s = dchunk % geo.dn_stages, n = dchunk / geo.dn_stages;
      if (n > 0 && !mbar_wait(&dempty[s], (n - 1) & 1, geo.wait_ns)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
        break;
      }
      unsigned char* st = arena + (size_t)s * geo.dn_stage;
      mbar_arrive_expect_tx(&dfull[s], code_bytes + 8u * I);
      bulk_g2s(st, pk.down_codes + ((size_t)e * H + (size_t)ht * kDnRows) * (I / 2), code_bytes,
               &dfull[s]);
      bulk_g2s(st + code_bytes,
               pk.down_scales + ((size_t)e * (H / 64) + 2 * (size_t)ht) * (4 * (size_t)I), 8u * I,
               &dfull[s]);
    }
    // do not leave while copies into this CTA's shared memory may still be in flight
    const int dused = dchunk < geo.dn_stages ? dchunk : geo.dn_stages;
    for (int i = 0; i < dused; ++i) {
      const int c2 = dchunk - 1 - i;
      (void)mbar_wait(&dfull[c2 % geo.dn_stages], (c2 / geo.dn_stages) & 1, geo.wait_ns);
    }
    return;
  }

  // ---------------- 3. gate/up + SiLU*up (consumer warps)
  const int g = lane >> 2, c = lane & 3;
  {
    int chunk = 0;
    const int jb_per_chunk = geo.KC / 128;
    for (int q = q0; q < q1; ++q) {
      const int gi = q / gu_tiles, it = q % gu_tiles;
      const DcGroup gm = grp[gi];
      const int slot0 = gm.slot0, n = gm.n;
      // this task's multipliers: the loads overlap the MMA loop
      const float mg = __ldg(&pk.mult[gm.expert * 3 + 0]);
      const float mu = __ldg(&pk.mult[gm.expert * 3 + 1]);
      const float sd = mode == 1 ? __ldg(&pk.down_in_scale[gm.expert]) : 0.0f;
      const float i6d = mode == 1 ? __ldg(&pk.down_inv6S[gm.expert]) : 0.0f;
      const bool gvalid = g < n;
      const int xrow = gvalid ? group_tok(gm.toks, g) : 0;
      const unsigned char* xr = xop + (size_t)xrow * geo.x_stride + c * 16;
      // two accumulator sets (alternate k-blocks of a warp): two independent MMA chains each
      float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
      float accg2[4] = {0.f, 0.f, 0.f, 0.f}, accu2[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kc = 0; kc < geo.nkc; ++kc, ++chunk) {
        const int s = chunk % geo.gu_stages, nn = chunk / geo.gu_stages;
        if (!abort_s && !mbar_wait(&gfull[s], nn & 1, geo.wait_ns)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        const unsigned char* st = arena + (size_t)s * geo.gu_stage;
        const unsigned char* scb = st + 32 * geo.row_bytes + c * 32 + g * 4;
        auto kblock = [&](int jb, float (&ag)[4], float (&au)[4]) {
          const int off = jb * 64 + c * 16;
          const uint4 gr = lds128(st + g * geo.row_bytes + off);
          const uint4 gr8 = lds128(st + (g + 8) * geo.row_bytes + off);
          const uint4 ur = lds128(st + (16 + g) * geo.row_bytes + off);
          const uint4 ur8 = lds128(st + (24 + g) * geo.row_bytes + off);
          const uint32_t scg = lds32(scb + jb * 128);
          const uint32_t scu = lds32(scb + geo.KC + jb * 128);
          uint4 xb[4];
          if (gvalid) {
            const unsigned char* xp = xr + (size_t)(kc * jb_per_chunk + jb) * 256;
#pragma unroll
            for (int p = 0; p < 4; ++p) xb[p] = lds128(xp + p * 64);
          } else {
#pragma unroll
            for (int p = 0; p < 4; ++p) xb[p] = make_uint4(0, 0, 0, 0);
          }
          kblock128_mma(ag, gr, gr8, scg, xb);
          kblock128_mma(au, ur, ur8, scu, xb);
        };
        for (int jb = warp; jb < jb_per_chunk; jb += 2 * kDcWarps) {
          kblock(jb, accg, accu);
          if (jb + kDcWarps < jb_per_chunk) kblock(jb + kDcWarps, accg2, accu2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gempty[s]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        accg[i] += accg2[i];
        accu[i] += accu2[i];
      }
      // partial sums of the 8 warps -> shared memory; 128 threads each finish one h element
      float* redq = red + (size_t)((q - q0) & (geo.redbufs - 1)) * (kDcWarps * 2 * 128);
      float* myred = redq + (size_t)(warp * 2) * 128;
      *reinterpret_cast<float4*>(myred + lane * 4) =
          make_float4(accg[0], accg[1], accg[2], accg[3]);
      *reinterpret_cast<float4*>(myred + 128 + lane * 4) =
          make_float4(accu[0], accu[1], accu[2], accu[3]);
      consumer_sync(kDcCons);
      if (tid < 128) {
        // thread = (column col, row r of the 16-row tile); the 16 rows of a column are 16
        // consecutive lanes. Accumulator element of (r, col): lane 4 (r % 8) + col / 2,
        // register (col % 2) + 2 (r / 8).
        const int col = tid >> 4, r = tid & 15;
        const int e_idx = (4 * (r & 7) + (col >> 1)) * 4 + (col & 1) + 2 * (r >> 3);
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int w = 0; w < kDcWarps; ++w) {
          gs += redq[(size_t)(w * 2) * 128 + e_idx];
          us += redq[(size_t)(w * 2) * 128 + 128 + e_idx];
        }
        const bool cvalid = col < n;
        const float xf = cvalid ? xfac_s[group_tok(gm.toks, col)] : 0.0f;
        const float hv = cvalid ? silu_mul(gs * mg * xf, us * mu * xf) : 0.0f;
        const size_t slot = (size_t)(slot0 + (cvalid ? col : 0));
        unsigned long long* htp = ws.htag + (slot * (I / 16) + it) * 9;
        if (mode == 0) {
          const uint16_t hb = f32_to_bf16_rn(hv);
          // |h| of the BF16 values over the column's 16 rows, for the down stage's f16 scaling
          float a = fabsf(__uint_as_float((uint32_t)hb << 16));
#pragma unroll
          for (int off = 1; off < 16; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
          const uint32_t hb_next = __shfl_down_sync(0xFFFFFFFFu, (uint32_t)hb, 1);
          if (cvalid) {
            ws.h16[slot * I + it * 16 + r] = hb;
            // tagged for the down stage: BF16 pairs (rows r, r+1) and the block's max |h|
            if ((r & 1) == 0) st_tag(htp + r / 2, (uint32_t)hb | (hb_next << 16), ep);
            if (r == 0) st_tag(htp + 8, __float_as_uint(a), ep);
          }
        } else if (a8) {
          // W4A8: h -> E4M3 with the down matrix's scale (i6d = fl32(1/fl32(6 sd))), one byte per
          // element; rows 4w..4w+3 of a column (its 16 consecutive lanes) make tagged word w
          const uint32_t q8 = a8_encode(hv, i6d);
          uint32_t wv = q8 << (8 * (r & 3));
          wv |= __shfl_xor_sync(0xFFFFFFFFu, wv, 1);
          wv |= __shfl_xor_sync(0xFFFFFFFFu, wv, 2);
          if (cvalid) {
            ws.hq[slot * I + it * 16 + r] = static_cast<uint8_t>(q8);
            if ((r & 3) == 0) st_tag(htp + r / 4, wv, ep);
          }
        } else {
          // the quantiser Q of this 16-element block of h (down input scale)
          float a = fabsf(hv);
#pragma unroll
          for (int off = 1; off < 16; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
          const uint32_t sf = e4m3_encode_rn(__fmul_rn(a, i6d));
          uint32_t nib = 0;
          if (sf != 0u) {
            const float rr = __frcp_rn(__fmul_rn(e4m3_value_nonneg(sf), sd));
            nib = e2m1_encode_rn(__fmul_rn(hv, rr)) << (4 * (r & 7));
          }
#pragma unroll
          for (int off = 1; off < 8; off <<= 1) nib |= __shfl_xor_sync(0xFFFFFFFFu, nib, off);
          const uint32_t hi_word = __shfl_down_sync(0xFFFFFFFFu, nib, 8);
          if (cvalid && r == 0) {
            *reinterpret_cast<uint2*>(ws.hq + slot * (I / 2) + it * 8) = make_uint2(nib, hi_word);
            ws.hsf[slot * (I / 16) + it] = static_cast<uint8_t>(sf);
            st_tag(htp + 0, nib, ep);
            st_tag(htp + 1, hi_word, ep);
            st_tag(htp + 2, sf, ep);
          }
        }
      }
      // with two buffers no barrier here: the next task's partials go to the other buffer,
      // and its own partial barrier comes after this epilogue in every thread (the down phase
      // starts with one)
      if (geo.redbufs == 1) consumer_sync(kDcCons);
    }
  }

  // ---------------- 4. down (consumer warps): each task waits only for its own group's h
  {
    const int nkb = I / 64, ntile = I / 16;
    const uint32_t code_bytes = (uint32_t)kDnRows * (I / 2);
    int cur = -1, dchunk = 0;
    float md = 0.0f;
    for (int i = 0; i < nd; ++i, ++dchunk) {
      const int q = dq(i);
      const int gi = q / dn_tiles, ht = q % dn_tiles;
      const DcGroup gm = grp[gi];
      const int slot0 = gm.slot0, n = gm.n;
      if (gi != cur) {
        // the group's h rows as the f16 operand: BF16 h * 2^-s (W4A16; s from the slot's
        // max |h|, exact) or the decoded NVFP4 code * scale (W4A4, exact). One (row, 16-block)
        // per thread: poll its tagged words, then convert.
        if (tid < kGroup) hamax_s[tid] = 0u;
        consumer_sync(kDcCons);
        md = __ldg(&pk.mult[gm.expert * 3 + 2]);
        const float sd = mode == 1 ? __ldg(&pk.down_in_scale[gm.expert]) : 0.0f;
        const int nent = n * ntile;
        if (mode == 0 && n == 1 && nent <= 32) {
          // one slot with at most 32 blocks: warp 0 polls its blocks, takes the slot's max |h|
          // by a warp reduction and converts in registers
          if (warp == 0) {
            unsigned long long w[9];
            uint32_t am = 0u;
            if (lane < nent) {
              if (!poll_tags<9>(ws.htag + ((size_t)slot0 * ntile + lane) * 9, ep, w, geo.wait_ns)) {
                record_status(ws.ctl, kStTimeout);
                abort_s = 1;
              }
              am = data_of(w[8]);
            }
            am = __reduce_max_sync(0xFFFFFFFFu, am);   // non-negative floats order as bits
            const int sh = amax_shift(__uint_as_float(am));
            const float f = pow2f(-sh);
            if (lane == 0) hfac_s[0] = pow2f(sh);
            if (lane < nent) {
              uint32_t* dst = reinterpret_cast<uint32_t*>(xop) + lane * 8;
#pragma unroll
              for (int p2 = 0; p2 < 8; ++p2) {
                const uint32_t v = data_of(w[p2]);
                const __half2 hh = __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), f),
                                                     __fmul_rn(__uint_as_float(v & 0xFFFF0000u), f));
                dst[p2] = *reinterpret_cast<const uint32_t*>(&hh);
              }
            }
          }
          consumer_sync(kDcCons);
          cur = gi;
        }
        for (int ent = tid; ent < nent && cur != gi; ent += kDcCons) {
          const int row = ent / ntile, it = ent % ntile;
          const unsigned long long* src = ws.htag + ((size_t)(slot0 + row) * ntile + it) * 9;
          unsigned long long w[9];
          bool ok;
          if (mode == 0) {
            ok = poll_tags<9>(src, ep, w, geo.wait_ns);
          } else if (a8) {
            unsigned long long w4[4];
            ok = poll_tags<4>(src, ep, w4, geo.wait_ns);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) w[q4] = w4[q4];
          } else {
            unsigned long long w3[3];
            ok = poll_tags<3>(src, ep, w3, geo.wait_ns);
            w[0] = w3[0];
            w[1] = w3[1];
            w[2] = w3[2];
          }
          if (!ok) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          uint32_t* dst = reinterpret_cast<uint32_t*>(xop + (size_t)row * geo.h_stride) + it * 8;
          if (mode == 0) {
            // raw BF16 pairs for now; converted once the row's max |h| is known
#pragma unroll
            for (int p2 = 0; p2 < 8; ++p2) dst[p2] = data_of(w[p2]);
            atomicMax(&hamax_s[row], data_of(w[8]));
          } else if (a8) {
            // W4A8: the E4M3 codes' values (exact in f16); the scale fl32(6 sd) in the epilogue
#pragma unroll
            for (int p2 = 0; p2 < 8; ++p2)
              dst[p2] = e4m3x2_to_f16x2(data_of(w[p2 >> 1]) >> (16 * (p2 & 1)));
            if (it == 0) hfac_s[row] = __fmul_rn(6.0f, sd);
          } else {
            const float sv = e4m3_value_nonneg(data_of(w[2]));
            const uint32_t cw[2] = {data_of(w[0]), data_of(w[1])};
#pragma unroll
            for (int p2 = 0; p2 < 8; ++p2) {
              const uint32_t byte = (cw[p2 >> 2] >> (8 * (p2 & 3))) & 0xFFu;
              const __half2 hh = __floats2half2_rn(e2m1_value(byte & 0xF) * sv,
                                                   e2m1_value(byte >> 4) * sv);
              dst[p2] = *reinterpret_cast<const uint32_t*>(&hh);
            }
            if (it == 0) hfac_s[row] = sd;
          }
        }
        if (cur != gi) consumer_sync(kDcCons);
        if (mode == 0 && cur != gi) {
          for (int ent = tid; ent < nent; ent += kDcCons) {
            const int row = ent / ntile, it = ent % ntile;
            const int sh = amax_shift(__uint_as_float(hamax_s[row]));
            const float f = pow2f(-sh);
            if (it == 0) hfac_s[row] = pow2f(sh);
            uint32_t* dst = reinterpret_cast<uint32_t*>(xop + (size_t)row * geo.h_stride) + it * 8;
#pragma unroll
            for (int p2 = 0; p2 < 8; ++p2) {
              const uint32_t v = dst[p2];
              const __half2 hh = __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), f),
                                                   __fmul_rn(__uint_as_float(v & 0xFFFF0000u), f));
              dst[p2] = *reinterpret_cast<const uint32_t*>(&hh);
            }
          }
          consumer_sync(kDcCons);
        }
        cur = gi;
      }
      const int s = dchunk % geo.dn_stages, nn = dchunk / geo.dn_stages;
      if (!abort_s && !mbar_wait(&dfull[s], nn & 1, geo.wait_ns)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      const unsigned char* st = arena + (size_t)s * geo.dn_stage;
      const bool gvalid = g < n;
      const unsigned char* hr = xop + (size_t)(gvalid ? g : 0) * geo.h_stride + c * 32;
      const unsigned char* rg = st + (size_t)(warp * 16 + g) * (I / 2) + c * 8;
      const unsigned char* rg8 = rg + 8 * (I / 2);
      const unsigned char* scb = st + code_bytes + (size_t)(warp >> 2) * (4 * I) +
                                 (size_t)(warp & 3) * nkb * 64 + c * 16 + g * 2;
      // two accumulators (even / odd k-blocks): two independent MMA chains
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
      auto dblock = [&](int j, float (&a)[4]) {
        const uint2 a0 = lds64(rg + j * 32);
        const uint2 a1 = lds64(rg8 + j * 32);
        const uint32_t sc = lds16(scb + j * 64);
        uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = xb0;
        if (gvalid) {
          xb0 = lds128(hr + j * 128);
          xb1 = lds128(hr + j * 128 + 16);
        }
        kblock_mma(a, a0, a1, sc, xb0, xb1);
      };
      for (int j = 0; j < nkb; j += 2) {
        dblock(j, acc);
        if (j + 1 < nkb) dblock(j + 1, acc2);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[s]);
      // Y = BF16(acc * md * factor): plain (slot-major rows) and tagged pairs of rows (r, r+1),
      // r even, for the combine; row g's partner g+1 is the lane 4 above
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const int col = 2 * c + (q2 & 1);
        const int row = ht * kDnRows + warp * 16 + g + ((q2 >> 1) << 3);
        const uint16_t yb = f32_to_bf16_rn(acc[q2] * md * hfac_s[col < n ? col : 0]);
        const uint32_t yb_next = __shfl_down_sync(0xFFFFFFFFu, (uint32_t)yb, 4);
        if (col < n && (g & 1) == 0) {
          // rows (row, row + 1) as one pair: plain (4-byte store) and tagged
          const size_t slot = (size_t)(slot0 + col);
          const uint32_t pair = (uint32_t)yb | (yb_next << 16);
          *reinterpret_cast<uint32_t*>(ws.y + slot * H + row) = pair;
          st_tag(ws.ytag + slot * (H / 2) + row / 2, pair, ep);
        }
      }
    }
  }

  // ---------------- 5. combine: 128-row tile ht of out is formed by the CTA of rank ht (mod
  // the grid) in the order (late down tasks, b) once
  // all of its Y pairs carry this epoch: the fixed-order weighted sum over each token's k
  // experts (rank order, FP32, then BF16)
  {
    uint32_t* ysm = reinterpret_cast<uint32_t*>(arena);   // [T][k][64] BF16 pairs of the tile
    for (int ht = sp.crank; ht < dn_tiles; ht += G) {
      consumer_sync(kDcCons);
      // 8 pairs per thread in flight at a time: (selection sj, pair p2) = it2 + u * 256
      for (int base = 0; base < S * 64; base += 8 * kDcCons) {
        unsigned long long w[8];
        bool have[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int it2 = base + tid + u * kDcCons;
          have[u] = it2 < S * 64;
          w[u] = have[u] ? ld_tag(ws.ytag + (size_t)sel_slot[it2 >> 6] * (H / 2) + ht * 64 +
                                  (it2 & 63))
                         : 0ull;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int it2 = base + tid + u * kDcCons;
          if (have[u]) ysm[it2] = data_of(w[u]);
        }
        // words that had not arrived yet: poll all of them together (one round trip per pass,
        // bounded)
        uint32_t late = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) late |= (have[u] && tag_of(w[u]) != ep) ? 1u << u : 0u;
        if (late) {
          const uint64_t t0 = globaltimer_ns();
          while (late) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (late & (1u << u)) {
                const int it2 = base + tid + u * kDcCons;
                w[u] = ld_tag(ws.ytag + (size_t)sel_slot[it2 >> 6] * (H / 2) + ht * 64 + (it2 & 63));
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if ((late & (1u << u)) && tag_of(w[u]) == ep) {
                ysm[base + tid + u * kDcCons] = data_of(w[u]);
                late &= ~(1u << u);
              }
            }
            if (late && globaltimer_ns() - t0 > geo.wait_ns) {
              record_status(ws.ctl, kStTimeout);
              abort_s = 1;
              break;
            }
          }
        }
      }
      consumer_sync(kDcCons);
      for (int it2 = tid; it2 < T * 64; it2 += kDcCons) {
        const int t = it2 >> 6, p2 = it2 & 63;
        float a0 = 0.0f, a1 = 0.0f;
        for (int j = 0; j < k; ++j) {
          const float wj = sel_w[t * k + j];
          const uint32_t v = ysm[(t * k + j) * 64 + p2];
          a0 += wj * __uint_as_float(v << 16);
          a1 += wj * __uint_as_float(v & 0xFFFF0000u);
        }
        if (SH) {
          // the shared expert's term, after the routed ones (computed in this launch: its
          // tagged gate and Ys words): sigma_t * BF16(Ys), Ys rounded like a routed expert's
          // output
          const unsigned long long* stag = ws.sh_tag + (size_t)T * sv.Is;
          unsigned long long wy[2], wg[1];
          if (!poll_tags<2>(stag + T + (size_t)t * H + ht * 128 + 2 * p2, ep, wy, geo.wait_ns) ||
              !poll_tags<1>(stag + t, ep, wg, geo.wait_ns)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          const float sg = __uint_as_float(data_of(wg[0]));
          a0 += sg * bf16_round(__uint_as_float(data_of(wy[0])));
          a1 += sg * bf16_round(__uint_as_float(data_of(wy[1])));
        } else if (ws.sh_y) {
          // the shared expert's term, after the routed ones (written by an earlier kernel):
          // sigma_t * BF16(Ys), Ys rounded like a routed expert's output
          const float sg = __ldcg(ws.sh_sigma + t);
          const float2 ys = __ldcg(reinterpret_cast<const float2*>(ws.sh_y + (size_t)t * H) +
                                   ht * 64 + p2);
          a0 += sg * bf16_round(ys.x);
          a1 += sg * bf16_round(ys.y);
        }
        const uint32_t pair =
            (uint32_t)f32_to_bf16_rn(a0) | ((uint32_t)f32_to_bf16_rn(a1) << 16);
        reinterpret_cast<uint32_t*>(out + (size_t)t * H)[ht * 64 + p2] = pair;
        if (xnext) {
          // a chained layer: the next layer's input is this layer's input plus its output (the
          // residual stream), BF16(x + out)
          const size_t w = (size_t)t * (H / 2) + ht * 64 + p2;
          const uint32_t xv = __ldg(reinterpret_cast<const uint32_t*>(x) + w);
          reinterpret_cast<uint32_t*>(xnext)[w] =
              (uint32_t)f32_to_bf16_rn(bf16_lo(xv) + bf16_lo(pair)) |
              ((uint32_t)f32_to_bf16_rn(bf16_hi(xv) + bf16_hi(pair)) << 16);
        }
      }
    }
  }

  if (b == 0) {
    // CTA 0 publishes the routing once its own work is done (no later phase reads it):
    // counts/offsets of every expert (binary search in the sorted selections), the per-token
    // experts, weights and slots, and the permutation
    for (int e = tid; e < E; e += kDcCons) {
      int lo = 0, hi = S;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sorted_e[mid] < e) lo = mid + 1; else hi = mid;
      }
      int lo2 = lo, hi2 = S;
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2) >> 1;
        if (sorted_e[mid] <= e) lo2 = mid + 1; else hi2 = mid;
      }
      ws.offsets[e] = lo;
      ws.counts[e] = lo2 - lo;
    }
    if (tid < S) {
      ws.idx[tid] = sel_idx[tid];
      ws.w[tid] = sel_w[tid];
      ws.slot_of[tid] = sel_slot[tid];
      ws.perm[sel_slot[tid]] = tid / k;
    }
    if (tid == 0) {
      ws.offsets[E] = S;
      ws.ctl[kCtlGroups] = (uint32_t)U;
      ws.ctl[kCtlUnique] = (uint32_t)U;
    }
  }

  // ---------------- the last CTA of the call publishes its epoch (after every CTA read it)
  consumer_sync(kDcCons);
  if (tid == 0 && (ticket_acq_rel(&ws.ctl[kCtlDone]) + 1u) % (uint32_t)G == 0u)
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(&ws.ctl[kCtlEpoch]), "r"(ep)
                 : "memory");
}


}  // namespace

// Geometry of the fused kernel for a shape, or false when it does not fit one SM's shared
// memory (the multi-kernel path serves such shapes).
bool decode_geom(int T, int H, int E, int k, int I, int num_ctas, void* out_geom) {
  DcGeom g{};
  g.wait_ns = kWaitLimitNs;
  g.skip_logits_cta = -1;
  g.sh_off = 0;
  g.sh_hs = 0;
  if (T < 1 || T > kNarrowT || num_ctas < 1) return false;
  g.rows_max = (E + num_ctas - 1) / num_ctas;
  if (g.rows_max > kDcWarps) return false;
  g.rs = 2 * H + 16;
  if (H % (kDcWarps * 32)) return false;            // whole k-step pairs per warp
  g.KC = H <= 4096 ? H : 4096;
  while (H % g.KC) g.KC -= 128;
  g.nkc = H / g.KC;
  g.row_bytes = g.KC / 2;
  g.gu_stage = 32 * g.row_bytes + 2 * g.KC;
  g.dn_stage = kDnRows * (I / 2) + 8 * I;
  g.x_stride = 2 * H + 64;
  g.h_stride = 2 * I + 16;
  g.xop = T * g.x_stride > kGroup * g.h_stride ? T * g.x_stride : kGroup * g.h_stride;
  g.smax = T * k;
  g.gmax = g.smax < E ? g.smax : E;
  g.xsep = T == 1 ? g.rs : 0;
  const int route_bytes = (g.rows_max + (g.xsep ? 0 : T)) * g.rs;
  const int scratch = T * k * 64 * 4;  // Y pairs of one tile for the combine
  const int red1 = kDcWarps * 2 * 128 * 4;   // one K-partial buffer
  int fixed = g.xop + red1 + g.gmax * (int)sizeof(DcGroup) + g.smax * 20 + 8 +
              8 * (2 * 3 + 2 * 16 + 3) + 16 + g.xsep + kDcStatic;
  g.redbufs = 1;
  if ((kDcSmemMax - fixed - red1) / g.gu_stage >= 2) {
    g.redbufs = 2;
    fixed += red1;
  }
  const int avail = kDcSmemMax - fixed;
  g.gu_stages = avail / g.gu_stage;
  if (g.gu_stages > 3) g.gu_stages = 3;
  if (g.gu_stages < 1) return false;
  int arena = g.gu_stages * g.gu_stage;
  if (arena < route_bytes) arena = route_bytes;
  if (arena < scratch) arena = scratch;
  if (arena > avail) return false;
  g.dn_stages = arena / g.dn_stage;
  if (g.dn_stages > 16) g.dn_stages = 16;
  if (g.dn_stages < 1) return false;
  g.arena = (arena + 127) & ~127;
  g.smem = g.arena + fixed - kDcStatic;
  if (g.smem + kDcStatic > kDcSmemMax) return false;
  if (out_geom) *static_cast<DcGeom*>(out_geom) = g;
  return true;
}

cudaError_t launch_decode(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                          float xS, float x_inv6S, const uint16_t* x, const uint16_t* wr,
                          uint16_t* out, uint16_t* xnext, const ShView* sv) {
  const int a8 = mode == 2;
  if (a8) mode = 1;   // W4A8 runs the quantised-activation instantiations
  DcGeom geo;
  if (!decode_geom(ws.T, ws.H, ws.E, ws.k, ws.I, lc.num_sms, &geo)) return cudaErrorInvalidValue;
  ShView svv{};
  int shf = 0;
  if (sv) {
    // the shared expert's gate/up rows of one CTA (2 rows of H BF16 per index) go into the
    // arena past the first gate/up stage and the staged router / activation rows
    if (ws.T > 2 || !ws.sh_tag || sv->Is % 64 != 0) return cudaErrorNotSupported;
    const int idx_max = (sv->Is + 1 + lc.num_sms - 1) / lc.num_sms;
    const int route_bytes = (geo.rows_max + (geo.xsep ? 0 : ws.T)) * geo.rs;
    int off = geo.gu_stage > route_bytes ? geo.gu_stage : route_bytes;
    off = (off + 127) & ~127;
    const long long hs_off = ((long long)off + (long long)idx_max * 2 * ws.H * 2 + 15) & ~15LL;
    if (hs_off + (long long)ws.T * sv->Is * 2 > geo.arena) return cudaErrorNotSupported;
    geo.sh_off = off;
    geo.sh_hs = (int)hs_off;
    svv = *sv;
    shf = 1;
  }
  const FaultInjection& fi = fault_injection();
  if (fi.wait_ns) geo.wait_ns = fi.wait_ns;
  geo.skip_logits_cta = fi.skip_logits_cta;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, geo.smem);
    if (e != cudaSuccess) return e;
    // the CTAs poll each other's results, so every one of them must be resident at once: one
    // CTA per SM must fit (else the caller takes the multi-kernel path)
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDcThreads, geo.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    return launch_kernel(lc, kern, dim3(lc.num_sms), dim3(kDcThreads), (size_t)geo.smem, pk, ws,
                         geo, x, wr, xS, x_inv6S, out, xnext, a8, svv);
  };
  if (shf) {
    if (mode == 1) return ws.T == 1 ? go(k_decode<1, 1, true>) : go(k_decode<2, 1, true>);
    return ws.T == 1 ? go(k_decode<1, 0, true>) : go(k_decode<2, 0, true>);
  }
  if (mode == 1) {
    switch (ws.T) {
      case 1: return go(k_decode<1, 1, false>);
      case 2: return go(k_decode<2, 1, false>);
      case 3: return go(k_decode<3, 1, false>);
      case 4: return go(k_decode<4, 1, false>);
      case 5: return go(k_decode<5, 1, false>);
      case 6: return go(k_decode<6, 1, false>);
      case 7: return go(k_decode<7, 1, false>);
      default: return go(k_decode<8, 1, false>);
    }
  }
  switch (ws.T) {
    case 1: return go(k_decode<1, 0, false>);
    case 2: return go(k_decode<2, 0, false>);
    case 3: return go(k_decode<3, 0, false>);
    case 4: return go(k_decode<4, 0, false>);
    case 5: return go(k_decode<5, 0, false>);
    case 6: return go(k_decode<6, 0, false>);
    case 7: return go(k_decode<7, 0, false>);
    default: return go(k_decode<8, 0, false>);
  }
}

}  // namespace moe
