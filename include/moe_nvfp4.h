/* moe_nvfp4.h — C ABI of the GB300 (sm_103a) NVFP4 routed-expert MoE feed-forward library.
 *
 * The operation is the routed-expert MoE feed-forward step of a Qwen-style sparse model as
 * the pages describe it:
 *   - the model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix (bit-exact)", first
 *     paragraph (512 routed experts per layer, top-10) and section "What is bit-exact and what
 *     is quantized" (each routed expert matrix stored as E2M1 codes, one E4M3 scale per 16
 *     weights, an FP32 multiplier and an FP32 activation input scale per matrix; the router
 *     stored BF16);
 *   - the Infernix README, section "Activation precision" (routed experts run W4A4 with the
 *     checkpoint's calibrated input scales, or with 16-bit activations on the same 4-bit
 *     weights), and the release notes "Infernix windows-2026.10.11", section "Highlights"
 *     (narrow expert calls of up to eight columns; the down pass launched as a dependent of
 *     gate/up).
 * Readings taken where the pages are silent: the router keeps the k largest logits (equal
 * logits: the lower expert index first) and weights them by the softmax over those k logits;
 * an expert computes down(SiLU(gate x) * up x); h = SiLU(gate)*up is rounded to BF16 (W4A16)
 * or quantised to NVFP4 with the down matrix's input scale (W4A4); each expert output Y is
 * rounded to BF16; out = BF16(sum_j w_j * Y_j) summed in rank order j = 0..k-1 in FP32.
 *
 * Conventions for every entry point:
 *   - All tensors are row-major. "device" pointers must be device memory of the current
 *     device, 16-byte aligned. BF16 tensors are passed as uint16_t bit patterns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; 0 = legacy default stream). No call
 *     except moe_pack_nvfp4 / moe_pack_destroy / moe_pack_get_matrix / moe_read_device_status
 *     allocates, frees or synchronises.
 *   - Argument errors return before anything is launched. A launch failure returns
 *     MOE_ERR_CUDA. Faults during execution surface on the caller's next synchronisation.
 *   - Kernels never wait without bound: an internal wait that exceeds ~2 s records
 *     MOE_ERR_TIMEOUT in the workspace status word (see moe_read_device_status) and the kernel
 *     returns; the outputs of that call are then undefined.
 *   - The caller owns x, router weights, outputs and the workspace. The library owns a pack
 *     from moe_pack_nvfp4 until moe_pack_destroy.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* a null/misaligned pointer, a bad size, k > E, ...             */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. W4A4 with unequal x scales)  */
  MOE_ERR_OOM = 3,          /* device allocation failed (moe_pack_nvfp4 only)               */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed                          */
  MOE_ERR_TIMEOUT = 5,      /* a device-side wait gave up (reported via the status word)     */
  MOE_ERR_WORKSPACE = 6     /* the workspace is smaller than moe_workspace_size reported     */
} moe_status;

typedef enum {
  MOE_W4A16 = 0,  /* BF16 activations on NVFP4 weights ("--a16-activations" route)          */
  MOE_W4A4 = 1,   /* activations quantised to NVFP4 with the per-matrix input scale         */
  MOE_W4A8 = 2    /* activations quantised to FP8 E4M3 ("--a8-activations" route; reading:
                   * E4M3 round-to-nearest-even, saturating at 448, sign kept, one FP32 scale
                   * per matrix S8 = fl32(6 S) from the matrix's input scale S, so
                   * code = E4M3(fl32(v * fl32(1 / S8))), value = E4M3(code) * S8; x per gate/up
                   * matrix, h with the down matrix's scale). Runs on the fused narrow-call
                   * kernel and the wide tensor-core f16 path; other shapes return
                   * MOE_ERR_UNSUPPORTED. */
} moe_mode;

/* Opaque, device-resident, library-owned set of one layer's routed experts. */
typedef struct moe_expert_pack moe_expert_pack;

/* One NVFP4 matrix in checkpoint layout (model card, "What is bit-exact and what is
 * quantized"): rows x cols weights, cols being the reduction dimension.
 *   codes  [rows][cols/2] bytes; element (r, c) is the low nibble of byte (r, c/2) when c is
 *          even and the high nibble when c is odd; bit 3 of a nibble is the sign (E2M1).
 *   scales [rows][cols/16] E4M3 bytes; scale (r, b) applies to columns 16b..16b+15.
 *   decoded weight = E2M1(code) * E4M3(scale) * multiplier.
 *   input_scale: the FP32 activation scale of the matrix (W4A4); ignored in W4A16.
 * codes/scales may be host or device pointers; they are only read during moe_pack_nvfp4. */
typedef struct {
  const uint8_t* codes;
  const uint8_t* scales;
  float multiplier;
  float input_scale;
} moe_nvfp4_matrix;

/* Build a pack from num_experts experts, each given as gate [inter x hidden], up
 * [inter x hidden] and down [hidden x inter] matrices (arrays of num_experts descriptors).
 * The codes are kept bit for bit; the scales are re-laid out for the kernels (bit-preserving:
 * moe_pack_get_matrix returns the input bytes). Requirements: hidden % 128 == 0,
 * inter % 64 == 0, hidden <= 8192, inter <= 2048, 1 <= num_experts <= 1024, every multiplier
 * and input_scale finite and > 0. Allocates device memory (MOE_ERR_OOM on failure) and
 * synchronises `stream` before returning. On success *out owns that memory. */
moe_status moe_pack_nvfp4(const moe_nvfp4_matrix* gate, const moe_nvfp4_matrix* up,
                          const moe_nvfp4_matrix* down, int num_experts, int hidden, int inter,
                          void* stream, moe_expert_pack** out);

/* Free a pack (null is accepted). The pack must not be in use by queued work. */
moe_status moe_pack_destroy(moe_expert_pack* pack);

/* Sizes of a pack, and its device bytes. Any output pointer may be null. */
moe_status moe_pack_info(const moe_expert_pack* pack, int* num_experts, int* hidden,
                         int* inter, size_t* device_bytes);

/* Copy one matrix of one expert back in checkpoint layout (which: 0 gate, 1 up, 2 down) into
 * host buffers codes [rows][cols/2] and scales [rows][cols/16], plus its multiplier and input
 * scale. Synchronous. For tests of the bit-preserving repack. */
moe_status moe_pack_get_matrix(const moe_expert_pack* pack, int expert, int which,
                               uint8_t* codes, uint8_t* scales, float* multiplier,
                               float* input_scale);

/* Workspace bytes moe_forward needs for (pack, T, k, mode). The workspace must be zero-filled
 * before its first use; every call leaves its counters at zero again, so a workspace can be
 * reused by later calls (with any pack, T, k, mode whose size fits) without re-zeroing. The
 * library records the layout of the last call on each workspace (by its start address) and,
 * when a narrow call (T <= 8) follows a call of another layout, clears that call's
 * synchronisation words with a memset on the call's stream first. After a call that reported an
 * error through the status word, zero the workspace again. */
moe_status moe_workspace_size(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                              size_t* bytes);

/* Workspace bytes moe_route_topk needs (same zero-fill rule). */
moe_status moe_route_workspace_size(int T, int H, int E, int k, size_t* bytes);

/* Router, top-k, softmax weights, histogram and permutation (the first steps of the MoE
 * step; model card: BF16 router, 512 experts, top-10).
 *   x        device [T][H] BF16;  router_w device [E][H] BF16.
 *   idx      device [T][k] int32: the selected experts of each token, by descending logit.
 *   w        device [T][k] float: softmax of the selected logits (sums to 1 per token).
 *   counts   device [E] int32: slots routed to each expert.
 *   offsets  device [E+1] int32: exclusive prefix sum of counts.
 *   perm     device [T*k] int32: token ids grouped by expert (ascending expert, then token).
 * Logits are accumulated in FP32 from exact BF16 products. Requirements: 1 <= T <= 65536,
 * H % 128 == 0, H <= 8192, 1 <= k <= min(E, 32), E <= 1024. */
moe_status moe_route_topk(const uint16_t* x, const uint16_t* router_w, int T, int H, int E,
                          int k, int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                          int32_t* perm, void* ws, size_t ws_bytes, void* stream);

/* moe_route_topk without a workspace argument, for callers that cannot allocate device memory:
 * runtimes whose allocator is frozen after start-up, and embedders that own no device allocator
 * (a plugin that is handed only its input and output buffers). The pages have no counterpart to
 * this entry point; it exists only for such callers. Arguments, outputs and requirements are
 * those of moe_route_topk. Its workspace is a fixed 4 MiB device array inside the library, held
 * by every GPU that loads the library until the process exits; shapes whose
 * moe_route_workspace_size exceeds 4 MiB return MOE_ERR_WORKSPACE before anything is launched.
 * No call allocates or frees memory. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and caches it; make that first call before any stream capture,
 * and do not use the entry point again after a cudaDeviceReset of that device in the same
 * process. Each call clears the array's control words (cudaMemsetAsync on `stream`) except the
 * status word: a device-side timeout of any call stays recorded until
 * moe_read_device_status(NULL, ...) reads and clears it. All calls share the one array: calls
 * that overlap on the GPU (e.g. on two streams) race, so the caller must serialise them. */
moe_status moe_route_topk_noalloc(const uint16_t* x, const uint16_t* router_w, int T, int H, int E,
                                  int k, int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                                  int32_t* perm, void* stream);

/* The whole MoE feed-forward step: out [T][H] BF16 (device) from x [T][H] BF16 and router_w
 * [E][H] BF16 (device), using the experts of `pack` in `mode`. T <= 8 runs the narrow decode
 * kernels; larger T runs the grouped (prefill) kernels. W4A4 and W4A8 require every gate and up
 * matrix of the pack to share one input scale (else MOE_ERR_UNSUPPORTED). out must not alias
 * x. ws/ws_bytes: see moe_workspace_size. */
moe_status moe_forward(const uint16_t* x, const uint16_t* router_w, const moe_expert_pack* pack,
                       int T, int k, moe_mode mode, uint16_t* out, void* ws, size_t ws_bytes,
                       void* stream);

/* The shared expert of a layer (model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix
 * (bit-exact)", section "What is bit-exact and what is quantized": shared experts and the
 * shared-expert gate are stored BF16; the card gives no formula, and the Qwen-style form is
 * taken). All pointers are caller-owned device memory, 16-byte aligned, BF16 bit patterns:
 *   gate_up [2*inter][hidden]: rows 0..inter-1 are the gate projection, inter..2*inter-1 up;
 *   down    [hidden][inter];
 *   gate    [hidden]: the gate vector; the token's weight is sigma_t = 1/(1 + exp(-x_t . gate)).
 * 64 <= inter <= 2048, inter % 64 == 0. The shared expert is BF16 in both modes. */
typedef struct {
  const uint16_t* gate_up;
  const uint16_t* down;
  const uint16_t* gate;
  int inter;
} moe_shared_expert;

/* Workspace bytes moe_forward_shared needs (same zero-fill rule as moe_workspace_size). */
moe_status moe_workspace_size_shared(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                                     int shared_inter, size_t* bytes);

/* moe_forward plus the shared expert: for token t,
 *   hs  = BF16( SiLU(Wg x_t) * (Wu x_t) ),   Ys = Wd hs   (FP32 accumulation),
 *   out[t] = BF16( sum_j w_j * Y_j  +  sigma_t * BF16(Ys) ),  the shared term added after the
 * routed ones in FP32; Ys is rounded to BF16 like each routed expert's output Y. Arguments and requirements are those of moe_forward, plus `shared` (above);
 * a null or invalid `shared` returns MOE_ERR_INVALID_ARG. For T <= 2 the shared expert is
 * computed inside the one launch of the routed step (one launch in all) when its gate/up rows fit
 * the kernel's shared memory; otherwise it runs first, as two CUDA-core GEMV kernels for
 * T <= 8 and as two tcgen05 BF16 GEMMs with a per-token kernel between them for larger T.
 * ws/ws_bytes: see moe_workspace_size_shared. */
moe_status moe_forward_shared(const uint16_t* x, const uint16_t* router_w,
                              const moe_expert_pack* pack, const moe_shared_expert* shared, int T,
                              int k, moe_mode mode, uint16_t* out, void* ws, size_t ws_bytes,
                              void* stream);

/* Byte offsets inside a moe_forward workspace of intermediate results, for tests:
 * the per-call routing tables and the quantised activations and h of the last call. */
typedef struct {
  size_t idx;        /* int32 [T][k]      */
  size_t w;          /* float [T][k]      */
  size_t counts;     /* int32 [E]         */
  size_t offsets;    /* int32 [E+1]       */
  size_t perm;       /* int32 [T*k]       */
  size_t slot_of;    /* int32 [T][k]: position of (t, idx[t][j]) in perm */
  size_t x_codes;    /* uint8 [T][H/2]   (W4A4: Q(x) codes, checkpoint nibble order;
                        W4A8: [T][H] E4M3 codes) */
  size_t x_scales;   /* uint8 [T][H/16]  (W4A4: Q(x) E4M3 scales)                    */
  size_t h_bf16;     /* uint16 [T*k][I]  (W4A16: h rounded to BF16, rows = perm slots) */
  size_t h_codes;    /* uint8 [T*k][I/2] (W4A4: Q(h) codes; W4A8: [T*k][I] E4M3 codes) */
  size_t h_scales;   /* uint8 [T*k][I/16] (W4A4: Q(h) scales)                        */
  size_t y;          /* uint16 [T*k][H]  BF16 expert outputs Y, rows = perm slots     */
} moe_ws_offsets;

moe_status moe_workspace_offsets(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                                 moe_ws_offsets* offsets);

/* Byte offsets inside a moe_forward_shared workspace of the shared expert's intermediate
 * results, for tests: h (uint16 BF16 [T][inter]), sigma (float [T]) and Y (float [T][hidden],
 * before its BF16 rounding, which the combine applies). The routed results sit at the offsets
 * moe_workspace_offsets gives. Any output pointer may be null. */
moe_status moe_workspace_offsets_shared(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                                        int shared_inter, size_t* h, size_t* sigma, size_t* y);

/* Workspace bytes moe_forward_layers needs for `layers` layers shaped like `pack` (same
 * zero-fill rule as moe_workspace_size): the control words and one region per layer. */
moe_status moe_workspace_size_layers(const moe_expert_pack* pack, int layers, int T, int k,
                                     moe_mode mode, size_t* bytes);

/* Offsets of layer `layer`'s intermediate results inside a moe_forward_layers workspace (as
 * moe_workspace_offsets for a single call), for tests. */
moe_status moe_workspace_offsets_layers(const moe_expert_pack* pack, int layers, int T, int k,
                                        moe_mode mode, int layer, moe_ws_offsets* offsets);

/* The MoE step of `layers` consecutive layers of a stack, chained through the residual stream:
 * layer 0 reads x [T][H]; layer l + 1 reads x_{l+1} = BF16(x_l + out_l), layer l's input plus
 * its output, as a decoder layer adds its MoE output to the residual stream (a reading: the
 * pages chain the layers of the stack but print no formula; attention and norms between the
 * MoE steps are not part of this library). As the release notes "Infernix windows-2026.10.11",
 * section "Highlights", chain the expert passes by programmatic dependent launch, each layer
 * is one launch chained to the previous one: for narrow calls (T <= 8) the fused kernel copies
 * its router rows before it waits for the previous layer and its combine also writes the
 * residual sum; other shapes run moe_forward's launch sequence per layer plus the residual sum.
 * The whole call can be captured in a CUDA graph.
 *   x         device [T][H] BF16, the first layer's input.
 *   router_w  host array of `layers` device pointers, router_w[l] [E][H] BF16.
 *   packs     host array of `layers` packs with equal hidden, inter and expert counts.
 *   out       device [layers][T][H] BF16: out[l] is layer l's MoE output (moe_forward of x_l);
 *             must not overlap x.
 * Every layer's output equals moe_forward's on the same input, bit for bit. W4A4 requires each
 * pack's gate/up input scales to be equal (else MOE_ERR_UNSUPPORTED).
 * ws/ws_bytes: see moe_workspace_size_layers. */
moe_status moe_forward_layers(const uint16_t* x, const uint16_t* const* router_w,
                              const moe_expert_pack* const* packs, int layers, int T, int k,
                              moe_mode mode, uint16_t* out, void* ws, size_t ws_bytes,
                              void* stream);

/* NVFP4 quantiser Q (test hook, also usable to build checkpoints): rows x cols BF16 values
 * (device, cols % 16 == 0) -> codes [rows][cols/2] and E4M3 scales [rows][cols/16] (device),
 * with per-matrix FP32 scale S = input_scale (> 0, finite). Steps, per 16-element block:
 * inv6S = fl32(1/fl32(6 S)); sf = E4M3_RNE_satfinite(fl32(amax * inv6S)); sf == 0 -> codes +0;
 * otherwise r = fl32(1/fl32(sf * S)) and q = E2M1_RNE_satfinite(fl32(v * r)) (ties to even,
 * sign kept, so negative values rounding to zero encode as -0). */
moe_status moe_quantize_act_nvfp4(const uint16_t* x, int rows, int cols, float input_scale,
                                  uint8_t* codes, uint8_t* scales, void* stream);

/* Read and clear the device status word of a workspace (synchronises `stream`). *status is
 * MOE_OK or the first error a kernel recorded (MOE_ERR_TIMEOUT). ws = NULL reads the status word
 * of moe_route_topk_noalloc's fixed array on the current device. */
moe_status moe_read_device_status(void* ws, void* stream, moe_status* status);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status status);

/* Number of CUDA kernels the last moe_forward / moe_forward_shared call on this host thread
 * launched. */
int moe_last_launch_count(void);

/* Profiling hook (measurement only; not needed for computing): for the NEXT moe_forward or
 * moe_forward_shared call on this host thread, record cudaEvent_t events[2i] before and
 * events[2i+1] after its i-th kernel launch on the call's stream (count <= 64 events, i.e. up to
 * 32 launches; later launches are not recorded). While profiling, the launches are not
 * overlapped by programmatic dependent launch. No other entry point may be called on this
 * thread between arming and that call. count = 0 cancels. */
moe_status moe_profile_next_forward(void* const* events, int count);

/* Test-only fault injection (not needed for computing; process-wide, for failure-detection
 * tests that must not fault a GPU): skip_logits_cta >= 0 makes that CTA of the fused narrow-call
 * kernel publish no router logits, so every CTA's wait for them runs out; wait_limit_seconds
 * > 0 replaces that kernel's ~2 s wait bound (0 restores it; at most 10 s); the next
 * fail_pack_allocations device allocations of moe_pack_nvfp4 fail (MOE_ERR_OOM). A call whose
 * wait ran out finishes, records MOE_ERR_TIMEOUT in the workspace status word, and leaves the
 * workspace to be zeroed again. moe_test_inject_faults(-1, 0, 0) switches everything off. */
moe_status moe_test_inject_faults(int skip_logits_cta, double wait_limit_seconds,
                                  int fail_pack_allocations);

/* Name of the kernel of the i-th launch of the last profiled call (cudaFuncGetName; static
 * storage), or NULL. */
const char* moe_profile_kernel_name(int i);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
