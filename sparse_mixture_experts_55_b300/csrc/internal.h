// internal.h -- workspace layout and kernel launchers shared by the library's
// translation units (not part of the public ABI; see include/moe.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// Rows of every expert segment in the grouped buffers are padded to a
// multiple of this, so a 128-row MMA tile never straddles two experts.
constexpr int kSegPad = 128;
// Router blocks: kRouteThreads threads, each owning one 16-byte slice of d;
// a block routes route_tpb consecutive tokens (a multiple of kRouteGroup,
// sized so that the grid is about one wave) and writes one expert histogram.
constexpr int kRouteThreads = 512;
constexpr int kRouteGroup = 4;
// Tokens whose (token, slot) entries one grouping block ranks.
constexpr int kGroupTokens = 256;
// Batches up to this many tokens are routed and grouped by one block, which
// also clears the call's status words and counters (no memset before it).
constexpr int kSingleRouteT = 8;
// The down GEMM's epilogue forms y when its contraction is not split, and for
// batches up to this many tokens when it is.
constexpr int kFuseSplitT = 4;
constexpr int kMaxE = 32;
constexpr int kMaxK = 2;
// Status-word slots at the start of the workspace.
constexpr int kStatusInts = 8;
// Stages of a forward pass, as indexed in a stamps array (stamps.cuh).
enum Stage {
  ST_ROUTE = MOE_STAGE_ROUTE, ST_GROUP = MOE_STAGE_GROUP, ST_GATHER = MOE_STAGE_GATHER,
  ST_GATE_UP = MOE_STAGE_GATE_UP, ST_QUANT_H = MOE_STAGE_QUANT_H, ST_DOWN = MOE_STAGE_DOWN,
  ST_COMBINE = MOE_STAGE_COMBINE, ST_NORM = MOE_STAGE_NORM
};
constexpr int kNumStages = MOE_NUM_STAGES;
static_assert(kNumStages == 8, "one stamp pair per stage");

// Launch `kernel` on stream s; with pdl the launch may begin while the
// previous kernel in the stream finishes (programmatic dependent launch): the
// kernel must execute griddepcontrol.wait before it reads that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct WsLayout {
  // byte offsets into the workspace
  size_t status, tile_cnt, tok_cnt, tail_flag, idx, gate, blockcounts, offsets, poffsets, pos, perm_tok, perm_gate, xperm, hbuf,
      obuf, gu_part, xnorm;
  size_t xscale, habs, hq, hscale;  // e4m3 variant only (0 bytes otherwise)
  size_t ab, dye, dab, dxc, dl, dwg_part;  // training only (0 bytes otherwise)
  size_t tail_part;   // expert GEMMs' tail split: fp32 first halves (0 bytes when no GEMM is unsplit)
  int tail_slots;     // split tiles the scratch holds (per GEMM launch)
  int dwg_chunks;     // token chunks of the router-weight gradient's partial sums
  size_t total;
  size_t zero_bytes;  // bytes from `status` that every call clears (status word + split counters)
  int T, K;
  int TK;             // T*K: rows of the compact grouped buffers
  bool fuse_combine;  // the down GEMM's epilogue also forms y (tensor-core paths: unsplit, or T <= kFuseSplitT)
  int R;              // padded grouped rows (upper bound): T*K + E*(kSegPad-1), rounded up to kSegPad
  int S;              // split count over the contraction of the down projection
  int kb_per_split;
  int S_gu;           // split count over the contraction of the gate/up projection
  int kb_per_split_gu;
  int form;           // expert GEMM form: 0 multicast pairs, 1 CTA-pair MMA, 2 2x2 multicast tiles
  bool train;         // training layout (bf16): saved pre-activations and backward buffers
  int route_tpb;      // tokens per router block
  int n_route_blocks;
  bool route_single;  // T <= kSingleRouteT: one block routes, groups and clears the status and counters
};

// Split of one grouped GEMM's contraction into S ranges of kb_per_split
// 64-deep k-blocks.
struct SplitPlan {
  int S, kb_per_split;
};
// Chooses the split from a makespan model of the persistent GEMM: cluster
// units of work (an expert's tile pairs times S) spread over `clusters`
// co-resident 2-CTA clusters, each unit costing its k-blocks plus a fixed
// overhead, inflated by the fp32 partial-sum traffic a split adds
// (part_ratio = partial bytes per split / weight bytes).  S = 1 unless a
// split shortens the modelled time by at least 3%.
SplitPlan plan_splits(long long TK, int E, int n_tiles, int kb, int clusters, double part_ratio);
// train: also lay out the saved pre-activations and the backward buffers
// (and keep the gate/up contraction unsplit, which the saving epilogue needs).
// routing_only: the caller runs the routing kernels only (no fused-combine
// counters in front of the routing arrays).
WsLayout ws_layout(int T, int d, int f, int E, int K, int dtype, int num_sms, bool train = false,
                   bool routing_only = false);

struct Ptrs {
  int *status;
  int *tile_cnt;  // arrival counters of split gate/up tiles
  int *tok_cnt;   // [T, down n-tiles] slot arrivals of the fused combine
  int *tail_flag; // [2][tail_slots][2] arrivals on the tail split's first halves (gate/up, down)
  float *tail_part;  // [tail_slots][2][128][256] fp32 first halves of the tail split
  int32_t *idx;
  float *gate;
  int32_t *blockcounts, *offsets, *poffsets, *pos, *perm_tok;
  float *perm_gate;
  void *xperm, *hbuf;
  float *obuf;    // [S, T*K, d] gate-scaled expert outputs, unpadded grouped rows
  float *gu_part; // [S_gu, T*K, 2f] fp32 partial sums of the split gate/up projection
  void *xnorm;  // [T, d] normalised block input (moe_block_forward)
  // e4m3 variant: X_perm holds codes [R, d]; H stays bf16 [R, f] and is
  // re-quantised into hq [R, f] with one scale per row
  float *xscale;  // [R] scale of each grouped activation row
  float *habs;    // [R, gate/up n-tiles] max |bf16 H| per row and tile
  void *hq;       // [R, f] e4m3 codes of H
  float *hscale;  // [R] scale of each H row
  // training (bf16): saved by the forward, then the backward's buffers
  void *ab;         // [R, 2f] bf16 pre-activations a = X W1 | b = X W3
  void *dye;        // [R, d] bf16 gate * dy per grouped row (padding rows zero)
  void *dab;        // [R, 2f] bf16 dL/da | dL/db
  float *dxc;       // [T*K, d] dL/dX per unpadded grouped row
  float *dl;        // [T, E] dL/dlogits
  float *dwg_part;  // [dwg_chunks, d, E] partial sums of dL/dWg
  // profiling calls only: [2 * kNumStages] begin/end times of each stage
  // (stamps.cuh); null otherwise
  unsigned long long *stamps;
};
Ptrs carve(void *ws, const WsLayout &L);

// Streaming multiprocessors of the current device (148 if it cannot be read).
int sm_count_or_default();
// MOE_OK on an sm_103a device, MOE_ERR_UNSUPPORTED on another part,
// MOE_ERR_CUDA if the device cannot be queried.
int check_device();

// -------- routing.cu
cudaError_t launch_route(const void *x, const void *Wg, int T, int d, int E, int K, int dtype, unsigned flags,
                         const WsLayout &L, const Ptrs &P, cudaStream_t s);
cudaError_t launch_group(int T, int E, int K, const WsLayout &L, unsigned flags, const Ptrs &P, cudaStream_t s);
// Router then grouping.  L.route_single: one block, launched with programmatic
// dependent launch, that first waits for the previous work in the stream and
// clears the status words and counters itself (the caller enqueues no memset).
// Otherwise the status block must be zero at launch: one fused launch when
// T <= kGroupTokens (P.status[1] serves as its ticket counter), else the two
// kernels above.
cudaError_t launch_route_group(const void *x, const void *Wg, int T, int d, int E, int K, int dtype, unsigned flags,
                               const WsLayout &L, const Ptrs &P, cudaStream_t s);
// zero_pads: also zero the rows of padding (training forward)
cudaError_t launch_gather(const void *x, int T, int d, int E, int dtype, int R, const Ptrs &P, int num_sms,
                          cudaStream_t s, bool zero_pads);
cudaError_t launch_combine(void *y, int T, int d, int K, int S, int dtype, unsigned flags, const Ptrs &P,
                           int num_sms, cudaStream_t s);
cudaError_t launch_route_export(int T, int E, int K, const Ptrs &P, int32_t *idx, float *gate,
                                int32_t *perm_tok, int32_t *offsets, int32_t *pos, cudaStream_t s);
cudaError_t launch_rmsnorm(const void *x, void *out, int T, int d, float eps, int dtype, cudaStream_t s,
                           unsigned long long *stamps = nullptr);

// -------- gemm_tc.cu (bf16 tensor-core path)
// slot_of (host array of E entries, or null): expert e's matrices are slot
// slot_of[e] of banks holding n_slots matrices each (the expert cache);
// without it, slot e of banks of E.
// y: the layer output, formed by the down GEMM's epilogue when L.fuse_combine
// (then no combine kernel runs).
cudaError_t launch_expert_gemms_bf16(const void *W1, const void *W3, const void *W2, int d, int f, int E,
                                     const WsLayout &L, const Ptrs &P, void *y, unsigned flags, int num_sms,
                                     cudaStream_t s, const int *slot_of = nullptr, int n_slots = 0);

// -------- fp8.cu (e4m3 expert weights)
cudaError_t launch_quantize_weights_fp8(const void *W, int E, int K, int N, void *Wq, float *scales, cudaStream_t s);
cudaError_t launch_gather_quant(const void *x, int T, int d, int E, int R, const Ptrs &P, int num_sms,
                                cudaStream_t s);
cudaError_t launch_quant_h(int f, int E, int TK, int n_tiles, const Ptrs &P, int num_sms, cudaStream_t s);
// gemm_tc.cu, e4m3 operands: gate/up GEMM, H quantisation, down GEMM
cudaError_t launch_expert_gemms_fp8(const void *W1q, const float *s1, const void *W3q, const float *s3,
                                    const void *W2q, const float *s2, int d, int f, int E, const WsLayout &L,
                                    const Ptrs &P, void *y, unsigned flags, int num_sms, cudaStream_t s);

// -------- gemm_simt.cu (exact fp32 path)
// -------- backward.cu / gemm_bwd.cu (bf16, d and f multiples of 64)
cudaError_t launch_bwd_prep(const void *dy, int T, int d, int E, int K, int S, const WsLayout &L, const Ptrs &P,
                            int num_sms, cudaStream_t s);
// events (optional): recorded after each of the four products / after dx and after dWg
cudaError_t launch_bwd_gemms(const void *W1, const void *W3, const void *W2, void *dW1, void *dW3, void *dW2, int d,
                             int f, int E, bool accumulate, bool force_timeout, const WsLayout &L, const Ptrs &P,
                             int num_sms, cudaStream_t s, void *const *events);
cudaError_t launch_bwd_input(const void *x, const void *Wg, void *dx, void *dWg, int T, int d, int E, int K,
                             bool accumulate, const WsLayout &L, const Ptrs &P, int num_sms, cudaStream_t s,
                             void *const *events);

cudaError_t launch_expert_ffn_f32(const void *W1, const void *W3, const void *W2, int d, int f, int E,
                                  const WsLayout &L, const Ptrs &P, cudaStream_t s);

}  // namespace moe
