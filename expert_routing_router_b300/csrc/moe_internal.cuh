// moe_internal.cuh -- shared pieces of the CUDA library (never seen by callers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxGroups = 32;
constexpr int kChunk = 2048;  // assignments per dispatch chunk (counting / slot pass)
// Static scratch of moe_dispatch_noalloc: per-chunk histogram, n_chunks * E int32.
constexpr int kNoAllocHistInts = 65536;

// ---------------------------------------------------------------- host-side view
struct Cfg {
  int N, d, E, k, R, rank_map, score_fn, normalize, G, TG, F, Fs, act;
  float cf;
  int64_t A;       // N * k assignments
  int C;           // capacity (INT32 max = none)
  int n_chunks;    // ceil(A / kChunk)
  int act_bytes;   // 4 (fp32) or 2 (bf16)
  int mode;        // MOE_DISPATCH_PACKED or MOE_DISPATCH_CAPACITY_PADDED
  int64_t send_rows;  // rows of the send buffer: A (packed) or E * C (padded)
};

// Tensor-core router: padded sizes and the K slicing of its GEMM.
struct RouterPlan {
  int Epad, dpad, kb_per_split, nsplit;
  int n_acc, acc_cols;   // TMEM accumulators per CTA and columns per accumulator
  int stacked_n;         // 1: the three terms stacked along N (3*Epad <= 256), x read once;
                         // 0: stacked along K, x read once per term
  size_t ws_bytes;       // bf16 3-term split of the router weight (3 * Epad * dpad)
  size_t partial_bytes;  // fp32 partial logits [nsplit, N, Epad]
};
constexpr int kSmTarget = 148;  // SM count the router slicing is planned for

// Workspace carve-up (one layout serves every call).
struct WsLayout {
  size_t status;      // int32 device status word (0 = ok)
  size_t router_w;    // RouterPlan::ws_bytes
  size_t router_partial;  // RouterPlan::partial_bytes
  size_t chunk_hist;  // [n_chunks, E] int32
  size_t h;           // FFN intermediate: [A, F] then [N, Fs], act dtype
  size_t sched;       // reserved scratch
  size_t total;
};

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 16-byte read-only streaming load (data read once in the kernel).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace moe

// ---------------------------------------------------------------- launchers (host)
namespace moe {
cudaError_t launch_route(const Cfg& c, const void* x, const float* w_router, const float* b_router,
                         const float* sel_bias, float* logits, int32_t* topk_idx, float* topk_w,
                         void* ws_split, float* partial, int* status, cudaStream_t s);
RouterPlan router_plan(const Cfg& c);
cudaError_t launch_router_gemm(const Cfg& c, const RouterPlan& rp, const void* x,
                               const float* w_router, void* ws_split, float* partial, int* status,
                               cudaStream_t s);
cudaError_t launch_dispatch(const Cfg& c, const int32_t* topk_idx, const void* x, void* xperm,
                            int32_t* expert_counts, int32_t* kept_counts, int32_t* expert_start,
                            int32_t* rank_counts, int32_t* rank_offsets, int32_t* slot_of,
                            int32_t* perm_src, int32_t* num_kept, int32_t* chunk_hist,
                            cudaStream_t s);
cudaError_t launch_dispatch_noalloc(const Cfg& c, const int32_t* topk_idx, const void* x,
                                    void* xperm, int32_t* expert_counts, int32_t* kept_counts,
                                    int32_t* expert_start, int32_t* rank_counts,
                                    int32_t* rank_offsets, int32_t* slot_of, int32_t* perm_src,
                                    int32_t* num_kept, cudaStream_t s);
cudaError_t launch_ffn_simt(const Cfg& c, const void* xperm, const int32_t* expert_start,
                            const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                            const void* x, const void* shared_gate_up, const void* shared_down,
                            void* yperm, void* yshared, void* h, cudaStream_t s);
cudaError_t launch_ffn_tc(const Cfg& c, const void* xperm, const int32_t* expert_start,
                          const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                          const void* x, const void* shared_gate_up, const void* shared_down,
                          void* yperm, void* yshared, void* h, int* status, cudaStream_t s,
                          int stall_cta = -1, void* gu_save = nullptr);
// The same two GEMMs on SM pairs (tcgen05 cta_group::2, ffn_tc2.cu): the prefill path.
cudaError_t launch_ffn_tc2(const Cfg& c, const void* xperm, const int32_t* expert_start,
                           const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                           const void* x, const void* shared_gate_up, const void* shared_down,
                           void* yperm, void* yshared, void* h, int* status, cudaStream_t s,
                           void* gu_save = nullptr);
cudaError_t launch_ffn_tc_small(const Cfg& c, const void* xperm, const int32_t* expert_start,
                                const int32_t* kept_counts, const void* w_gate_up,
                                const void* w_down, const void* x, const void* shared_gate_up,
                                const void* shared_down, void* yperm, void* yshared, void* h,
                                int* status, cudaStream_t s);
// Average send-buffer rows per expert below which the token-major small-segment
// expert kernel is used (decode-sized batches).
#ifndef MOE_SMALL_ROWS
#define MOE_SMALL_ROWS 4
#endif
constexpr int kSmallRowsPerExpert = MOE_SMALL_ROWS;
// Average send-buffer rows per expert from which the SM-pair kernels (256-row tiles)
// are used for the expert FFN: below it, padding every expert's last tile to 256 rows
// costs more than the pair saves on the weight stream.
#ifndef MOE_PAIR_ROWS
#define MOE_PAIR_ROWS 512
#endif
constexpr int kPairRowsPerExpert = MOE_PAIR_ROWS;
cudaError_t launch_combine(const Cfg& c, const void* yperm, const int32_t* slot_of,
                           const float* topk_w, const void* residual, const void* yshared,
                           void* out, cudaStream_t s);
cudaError_t launch_bias_update(const Cfg& c, const int32_t* expert_counts, float* sel_bias,
                               float step, cudaStream_t s);
// INT8 payload (payload_q8.cu)
cudaError_t launch_dispatch_q8(const Cfg& c, const int32_t* topk_idx, const void* x, int8_t* xq,
                               float* xscale, int32_t* expert_counts, int32_t* kept_counts,
                               int32_t* expert_start, int32_t* rank_counts, int32_t* rank_offsets,
                               int32_t* slot_of, int32_t* perm_src, int32_t* num_kept,
                               int32_t* chunk_hist, cudaStream_t s);
cudaError_t launch_quant_rows(const Cfg& c, const void* in, const int32_t* perm_src, int8_t* q,
                              float* scale, cudaStream_t s);
cudaError_t launch_dequant_rows(const Cfg& c, const int8_t* q, const float* scale,
                                const int32_t* perm_src, void* out, cudaStream_t s);
cudaError_t launch_combine_q8(const Cfg& c, const int8_t* yq, const float* yscale,
                              const int32_t* slot_of, const float* topk_w, const void* residual,
                              const void* yshared, void* out, cudaStream_t s);
// backward (backward.cu, ffn_bwd_tc.cu)
cudaError_t launch_combine_backward(const Cfg& c, const void* dout, const void* yperm,
                                    const int32_t* slot_of, const float* topk_w, void* dyperm,
                                    float* dtopk_w, cudaStream_t s);
cudaError_t launch_route_backward(const Cfg& c, const void* x, const float* w_router,
                                  const float* logits, const int32_t* topk_idx,
                                  const float* dtopk_w, float* dlogits, float* dx_router,
                                  float* dw_router, float* db_router, void* ws, int* status,
                                  cudaStream_t s);
// The router's weight gradient on the tensor cores (router_bwd_tc.cu): dWr = dl^T x over
// a 3-term bf16 split of dl, db by a fixed-order column sum.  ws: router_bwd_ws_bytes.
size_t router_bwd_ws_bytes(const Cfg& c);
cudaError_t launch_router_dw_tc(const Cfg& c, const float* dlogits, const void* x, float* dw_router,
                                float* db_router, void* ws, int* status, cudaStream_t s);
// Tokens from which a bf16 layer's router weight gradient runs on the tensor cores.
constexpr int kRouterDwTcTokens = 128;
cudaError_t launch_dispatch_backward(const Cfg& c, const void* dxperm, const int32_t* slot_of,
                                     const void* dout, const void* dx_shared,
                                     const float* dx_router, void* dx, cudaStream_t s);
size_t ffn_backward_ws_bytes(const Cfg& c);
cudaError_t launch_ffn_backward(const Cfg& c, const void* xperm, const int32_t* expert_start,
                                const int32_t* kept_counts, const void* w_gate_up,
                                const void* w_down, const void* x, const void* shared_gate_up,
                                const void* shared_down, const void* dyperm, const void* dout,
                                void* dxperm, void* dx_shared, void* dw_gate_up, void* dw_down,
                                void* dshared_gate_up, void* dshared_down, const void* saved,
                                void* ws, int* status, cudaStream_t s);
// Bytes of the activations a training forward keeps for the backward:
// h [S, F] + [N, Fs], then g|u [S, 2F] + [N, 2Fs], bf16.
size_t saved_bytes(const Cfg& c);
int num_sms();

// Launch `kern` as a programmatic dependent of the kernel before it on stream `s`: its
// CTAs may be scheduled while that kernel still runs (once all of that kernel's CTAs
// have started and executed griddepcontrol.launch_dependents, or exited), so `kern`
// executes griddepcontrol.wait before it reads anything that kernel writes.  Outside a
// programmatic launch the wait returns at once.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
}  // namespace moe
