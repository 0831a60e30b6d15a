// Internal declarations shared by the library's translation units.
#pragma once

#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------- layout
// Device layout of one quantised matrix W [rows][K] (K = reduction axis,
// padded up to a multiple of 256 with zero-point codes and zero scales).
// Rows are taken in tiles of 16 and columns in blocks of 256: one (tile,
// block) is the weight operand of 16 consecutive mma.m16n8k16 steps.  Lane l
// of a warp owns 4*b words of each (tile, block): the codes of its A-fragment
// elements (rows l/4 and l/4 + 8; columns 2(l%4), +1, +8, +9 of each
// 16-column step), stored as bf16-pair fields so that one mask-and-or turns
// two codes into a bf16x2 register (see pair_bits in decode.cu).  Word q of
// lane l of (tile mt, block kb) sits at byte
//     ((mt * nkb + kb) * b + q / 4) * 512 + l * 16 + (q % 4) * 4,
// so each of a warp's b 16-byte loads per (tile, block) covers 512 contiguous
// bytes.  Scales: element (mt * ngroups + g) * 16 + r for row mt*16 + r and
// group g (ngroups counts the padded K).
constexpr int kTileRows = 16;
constexpr int kBlockK = 256;
constexpr int kBRows = 128;          // rows of the down projection per B work unit (8 row tiles)
constexpr int kDecodeMaxTokens = 8;  // forwards with T <= this use the decode path
constexpr int kMaxTopK = 8;
constexpr int kGroupChunk = 2048;  // prefill grouping: slots per bucket-pass block
constexpr int kWarps = 16;           // warps per CTA of the decode expert kernel

struct MatLayout {
  int rows, cols, kpad;  // cols = K; kpad = K rounded up to kBlockK
  int64_t codes_off, codes_bytes;
  int64_t scales_off, scales_bytes;
};

struct ExpertLayout {
  MatLayout m[3];      // 0 = gate [I][H], 1 = up [I][H], 2 = down [H][I]
  int64_t blob_bytes;  // bytes one expert occupies (padded K, sections 256-byte aligned)
  int64_t algo_bytes;  // codes + scales of the unpadded matrices: the algorithmic bytes
};

ExpertLayout make_layout(int H, int I, int bits, int group, int scale_dtype);

inline int scale_size(int dt) { return dt == MOE_SCALE_F32 ? 4 : 2; }

// Device counters per layer (uint64): order must match kStat*.
enum {
  kStatAccesses = 0, kStatHits, kStatMisses, kStatAdmissions, kStatEvictions, kStatHbmBytes,
  kStatHostBytes, kStatFillBytes, kStatPairs, kStatForwards, kStatRouterExact, kNumStats
};

// Error bits latched by kernels into the plan's error word.
enum : uint32_t { kErrTimeout = 1u, kErrBounds = 2u };

// Control words of the decode path (device).
struct Ctl {
  unsigned epoch;  // forward counter: bumped by the router kernel, tags the hand-off words
  int step;        // cache step: read by the forwards, advanced by the step-end kernel
  unsigned pad[6];
};

struct Plan {
  moe_plan_desc d{};
  ExpertLayout lay{};
  int sms = 0;
  int max_distinct = 0;  // bound on D for the decode path

  // arenas
  uint8_t* hbm_arena = nullptr;  // STATIC: experts; LFU: slots
  uint8_t* pf_arena = nullptr;   // prefill_slots staging slots of a chunked prefill
  const uint8_t** pf_blob = nullptr;  // [E] the chunked prefill's residence of one layer
  unsigned* pf_stage = nullptr;       // [2] counts, then [E] (expert, slot) pairs staged
  int64_t hbm_cap = 0, hbm_used = 0;
  uint8_t* host_arena = nullptr;      // pinned, mapped
  uint8_t* host_arena_dev = nullptr;  // its device alias
  int64_t host_cap = 0, host_used = 0;
  int numa_node = -1;      // the GPU's NUMA node the host arena was bound to (-1: none)

  // residence (device tables [L*E]) and host mirrors
  const uint8_t** blob_hbm = nullptr;
  const uint8_t** blob_host = nullptr;
  std::vector<int64_t> hbm_pos, host_pos;         // arena position or -1
  std::vector<int64_t> hbm_free;                  // HBM positions vacated by experts moved to host
  std::vector<const uint8_t*> tab_hbm, tab_host;  // host mirrors of blob_hbm / blob_host
  std::vector<uint8_t> placed;

  // routers
  std::vector<uint16_t*> wr;  // device [E][H] bf16 per layer
  std::vector<float*> bias;   // device [E] per layer (zeros when none), rows of bias_all
  float* bias_all = nullptr;  // device [L][E]
  float* wnorm_all = nullptr;  // device [L][E] upper bounds of the router rows' 2-norms
  // prefill routing: cuBLAS handle with a workspace of its own (no allocation in a forward)
  cublasHandle_t blas = nullptr;
  void* blas_ws = nullptr;
  int blas_status = 0;  // a failed cuBLAS call of the last prefill forward (reported, then cleared)
  static constexpr size_t kBlasWorkspace = size_t(32) << 20;

  // forward scratch (device)
  float* logits = nullptr;            // [maxT][E]
  int32_t* topk_idx = nullptr;        // [maxT][k]
  float* topk_w = nullptr;            // [maxT][k]
  int32_t* counts = nullptr;          // [E]
  int32_t* offsets = nullptr;         // [E+1]
  int32_t* perm = nullptr;            // [maxT*k]
  int32_t* inv = nullptr;             // [maxT*k]
  int32_t* wl_expert = nullptr;       // [maxD] distinct experts, host-resident first
  int32_t* wl_off = nullptr;          // [maxD] offset into perm
  int32_t* wl_cnt = nullptr;          // [maxD] tokens routed to it
  const uint8_t** wl_blob = nullptr;  // [maxD] where to read it
  Ctl* ctl = nullptr;
  // Hand-off words between CTAs of the decode expert kernel: 32-bit payload in
  // the low half, the forward's epoch in the high half (zeroed at creation).
  unsigned long long* hbuf = nullptr;  // [maxD][decode T][kpad(I)/2] bf16 pairs of h
  unsigned long long* obuf = nullptr;  // [decode T * k][H] fp32 weighted expert outputs per slot
  float* xsum = nullptr;        // [decode T][H / G] scale-group sums of the layer input
  uint16_t* pf_h = nullptr;     // prefill: [maxT * k][I] bf16 h per (expert, token) slot, perm order
  uint16_t* pf_o = nullptr;     // prefill: [maxT * k][H] bf16 weighted expert output per slot
  int32_t* pf_bucket = nullptr;  // prefill grouping: [E][chunks of kGroupChunk slots] counts, then bases
  uint16_t* x_stage = nullptr;  // [maxT][H] for the host-buffer forward
  uint16_t* y_stage = nullptr;

  // LFU cache state (device)
  int32_t* slot_of = nullptr;     // [L*E] slot or -1
  int32_t* slot_owner = nullptr;  // [C] global expert id or -1
  uint32_t* lfu_count = nullptr;  // [L*E]
  int32_t* lfu_last = nullptr;    // [L*E] last step accessed (-1 = never)
  int32_t* miss_list = nullptr;   // [L * maxD] misses of the current step
  unsigned* miss_count = nullptr;
  unsigned* adm_list = nullptr;   // step-end: admitted (expert, slot) pairs
  unsigned* adm_count = nullptr;
  int step = 0;  // host mirror of ctl->step (steps ended through the API)

  // statistics and errors
  unsigned long long* stats = nullptr;    // [L][kNumStats]
  volatile uint32_t* err_host = nullptr;  // mapped pinned word
  uint32_t* err_dev = nullptr;

  // streams
  cudaStream_t aux = nullptr;  // second stream (placement, host-resident experts)
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_done = nullptr;
  cudaStream_t last_stream = nullptr;
  bool have_last = false;

  // decode launch configuration per batch size T (computed on first use)
  struct DecodeCfg {
    bool ready = false;
    size_t smem = 0, rsmem = 0;
    int grid = 0, slot_bytes = 0, nslots = 0;
  } dcfg[kDecodeMaxTokens + 1];

  bool fail_next = false;  // test hook: the next decode forward publishes no gate/up results

  std::atomic<int> busy{0};
  std::string last_error;
};

// Makes `fn` launchable with `bytes` of dynamic shared memory on the current
// device.  The attribute belongs to the function, not to a plan, so it is only
// ever raised (process-wide, per device): lowering it for one plan would make
// another plan's larger launch of the same kernel fail.
cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes);

// Launchers implemented in the .cu files (return cudaError_t of the launch).
cudaError_t router_norms(const uint16_t* wr, int E, int H, float* out, cudaStream_t s);
cudaError_t launch_repack(const uint8_t* src_codes, const void* src_scales, uint8_t* dst_blob,
                          const MatLayout& m, int bits, int group, int scale_dtype,
                          cudaStream_t s);
cudaError_t launch_quantize(const float* w, int rows, int cols, int bits, int group, int sdt,
                            uint8_t* codes, void* scales, cudaStream_t s);
// res / ysum (both or neither): also ysum = bf16(y + res), res fp32 [T][H]
cudaError_t decode_forward(Plan& p, int layer, const uint16_t* x, int T, uint16_t* y,
                           cudaStream_t s, const moe_routing_out* dbg, const float* res = nullptr,
                           uint16_t* ysum = nullptr);
cudaError_t lfu_step_end(Plan& p, cudaStream_t s);
// lfu = false: the forward leaves the LFU state (counts, miss queue) as it is;
// blob_hbm: the layer's HBM residence table to read (nullptr: the plan's own).
cudaError_t prefill_forward(Plan& p, int layer, const uint16_t* x, int T, uint16_t* y, cudaStream_t s,
                            const moe_routing_out* dbg, bool lfu = true,
                            const uint8_t* const* blob_hbm = nullptr, const float* res = nullptr,
                            uint16_t* ysum = nullptr);
// Stages the layer's experts that are not in HBM into the prefill slots and
// builds p.pf_blob (stream-ordered).
cudaError_t prefill_stage(Plan& p, int layer, cudaStream_t s);

}  // namespace moe
