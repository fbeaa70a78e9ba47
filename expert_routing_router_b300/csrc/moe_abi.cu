// moe_abi.cu -- the extern "C" entry points declared in include/moe.h.
//
// Every call validates its arguments on the host, resolves the workspace layout,
// checks the device once (compute capability 10.3), then enqueues its kernels on
// the caller's stream.  Nothing here allocates device memory or synchronises.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "moe_internal.cuh"

namespace moe {

int num_sms() {
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 148;
  }
  return cached[dev];
}

namespace {

moe_status check_device() {
  static int ok[64];  // 0 unknown, 1 supported, 2 not supported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (ok[dev] == 0) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    ok[dev] = (maj == 10 && min == 3) ? 1 : 2;
  }
  return ok[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host-side view of the configuration, or an error.
moe_status make_cfg(const moe_config* in, Cfg* c) {
  if (!in) return MOE_ERR_INVALID_ARG;
  const moe_config& m = *in;
  if (m.tokens < 1 || m.hidden < 8 || m.hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (m.num_experts < 1 || m.num_experts > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (m.top_k < 1 || m.top_k > kMaxTopK || m.top_k > m.num_experts) return MOE_ERR_INVALID_ARG;
  if (m.num_ranks < 1 || m.num_ranks > m.num_experts) return MOE_ERR_INVALID_ARG;
  if (m.rank_map != MOE_RANK_CONTIGUOUS && m.rank_map != MOE_RANK_ROUND_ROBIN)
    return MOE_ERR_INVALID_ARG;
  if (m.rank_map == MOE_RANK_CONTIGUOUS && m.num_experts % m.num_ranks != 0)
    return MOE_ERR_INVALID_ARG;
  if (m.score_fn != MOE_SCORE_SOFTMAX && m.score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (m.num_groups < 1 || m.num_groups > kMaxGroups || m.num_experts % m.num_groups != 0)
    return MOE_ERR_INVALID_ARG;
  if (m.topk_groups < 1 || m.topk_groups > m.num_groups) return MOE_ERR_INVALID_ARG;
  if ((int64_t)m.topk_groups * (m.num_experts / m.num_groups) < m.top_k) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(m.capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (m.d_ff < 8 || m.d_ff % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (m.shared_d_ff < 0 || m.shared_d_ff % 8 != 0) return MOE_ERR_INVALID_ARG;
  // weight rows are addressed by 32-bit tensor-map coordinates
  if ((int64_t)m.num_experts * 2 * m.d_ff > INT32_MAX ||
      (int64_t)m.num_experts * m.hidden > INT32_MAX || 2 * (int64_t)m.shared_d_ff > INT32_MAX)
    return MOE_ERR_INVALID_ARG;
  if (m.act_dtype != MOE_DTYPE_F32 && m.act_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (m.dispatch_mode != MOE_DISPATCH_PACKED && m.dispatch_mode != MOE_DISPATCH_CAPACITY_PADDED)
    return MOE_ERR_INVALID_ARG;
  if (m.dispatch_mode == MOE_DISPATCH_CAPACITY_PADDED && !(m.capacity_factor > 0.0f))
    return MOE_ERR_INVALID_ARG;
  const int64_t A = (int64_t)m.tokens * m.top_k;
  if (A > INT32_MAX / 2) return MOE_ERR_INVALID_ARG;  // slots are int32
  c->N = m.tokens;
  c->d = m.hidden;
  c->E = m.num_experts;
  c->k = m.top_k;
  c->R = m.num_ranks;
  c->rank_map = m.rank_map;
  c->score_fn = m.score_fn;
  c->normalize = m.normalize_topk != 0;
  c->G = m.num_groups;
  c->TG = m.topk_groups;
  c->F = m.d_ff;
  c->Fs = m.shared_d_ff;
  c->act = m.act_dtype;
  c->cf = m.capacity_factor;
  c->A = A;
  c->act_bytes = m.act_dtype == MOE_DTYPE_F32 ? 4 : 2;
  c->n_chunks = (int)((A + kChunk - 1) / kChunk);
  // C = ceil(cf * N * k / E) in double; cf <= 0: no cap
  if (m.capacity_factor > 0.0f) {
    const double cap = std::ceil((double)m.capacity_factor * (double)m.tokens * (double)m.top_k /
                                 (double)m.num_experts);
    c->C = cap > (double)INT32_MAX ? INT32_MAX : (int)cap;
  } else {
    c->C = INT32_MAX;
  }
  c->mode = m.dispatch_mode;
  c->send_rows = A;
  if (c->mode == MOE_DISPATCH_CAPACITY_PADDED) {
    c->send_rows = (int64_t)c->C * m.num_experts;
    if (c->send_rows > INT32_MAX / 2) return MOE_ERR_INVALID_ARG;  // slots are int32
  }
  return MOE_OK;
}

size_t round_up(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout layout(const Cfg& c) {
  WsLayout w;
  size_t off = 0;
  w.status = off;
  off += 256;
  w.router_w = off;
  w.router_partial = off;
  if (c.act == MOE_DTYPE_BF16) {
    const RouterPlan rp = router_plan(c);
    off += round_up(rp.ws_bytes);
    w.router_partial = off;
    off += round_up(rp.partial_bytes);
  }
  w.chunk_hist = off;
  off += round_up((size_t)c.n_chunks * c.E * sizeof(int32_t));
  w.h = off;
  off += round_up(((size_t)c.send_rows * c.F + (size_t)c.N * c.Fs) * c.act_bytes);
  w.sched = off;
  off += round_up(16 * 1024);
  w.total = off;
  return w;
}

moe_status ws_check(const Cfg& c, void* ws, size_t bytes, WsLayout* w) {
  *w = layout(c);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (bytes < w->total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// stall_cta >= 0 (self-test only) runs the prefill tensor-core kernels with that CTA's
// first ring slot never loaded; otherwise the kernel is chosen by rows per expert.
moe_status expert_ffn_impl(const moe_config* cfg, const void* xperm, const int32_t* expert_start,
                           const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                           const void* x, const void* shared_gate_up, const void* shared_down,
                           void* yperm, void* yshared, void* workspace, size_t workspace_bytes,
                           void* stream, int stall_cta, void* saved = nullptr,
                           size_t saved_size = 0) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!xperm || !expert_start || !kept_counts || !w_gate_up || !w_down || !yperm)
    return MOE_ERR_INVALID_ARG;
  if (c.Fs > 0 && (!x || !shared_gate_up || !shared_down || !yshared)) return MOE_ERR_INVALID_ARG;
  const void* acts[] = {xperm, w_gate_up, w_down, yperm};
  for (const void* p : acts)
    if (!aligned(p, 16)) return MOE_ERR_INVALID_ARG;
  if (c.Fs > 0 && (!aligned(x, 16) || !aligned(shared_gate_up, 16) || !aligned(shared_down, 16) ||
                   !aligned(yshared, 16)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_start, 4) || !aligned(kept_counts, 4)) return MOE_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = ws_check(c, workspace, workspace_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  void* h = static_cast<char*>(workspace) + w.h;
  int* status = reinterpret_cast<int*>(static_cast<char*>(workspace) + w.status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* xs = c.Fs > 0 ? x : nullptr;
  if (saved) {  // training forward: h and g|u go to the caller's buffer (prefill kernels)
    if (c.act != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
    if (!aligned(saved, 16)) return MOE_ERR_INVALID_ARG;
    if (saved_size < saved_bytes(c)) return MOE_ERR_WORKSPACE;
    __nv_bfloat16* hs = static_cast<__nv_bfloat16*>(saved);
    __nv_bfloat16* gus = hs + (size_t)c.send_rows * c.F + (size_t)c.N * c.Fs;
    if (c.A >= (int64_t)kPairRowsPerExpert * c.E)
      return from_cuda(launch_ffn_tc2(c, xperm, expert_start, kept_counts, w_gate_up, w_down,
                                      xs, shared_gate_up, shared_down, yperm, yshared, hs, status,
                                      s, gus));
    return from_cuda(launch_ffn_tc(c, xperm, expert_start, kept_counts, w_gate_up, w_down, xs,
                                   shared_gate_up, shared_down, yperm, yshared, hs, status, s,
                                   -1, gus));
  }
  if (stall_cta >= 0) {
    if (c.act != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
    return from_cuda(launch_ffn_tc(c, xperm, expert_start, kept_counts, w_gate_up, w_down, xs,
                                   shared_gate_up, shared_down, yperm, yshared, h, status, s,
                                   stall_cta));
  }
  if (c.act == MOE_DTYPE_F32)
    return from_cuda(launch_ffn_simt(c, xperm, expert_start, kept_counts, w_gate_up, w_down, xs,
                                     shared_gate_up, shared_down, yperm, yshared, h, s));
  // few rows per expert (decode): token-major kernel with right-sized token loads
  if (c.A < (int64_t)kSmallRowsPerExpert * c.E)
    return from_cuda(launch_ffn_tc_small(c, xperm, expert_start, kept_counts, w_gate_up, w_down,
                                         xs, shared_gate_up, shared_down, yperm, yshared, h,
                                         status, s));
  // many rows per expert: 256-row tiles on SM pairs (half the weight stream per SM);
  // otherwise 128-row tiles on single SMs (less padding of each expert's last tile)
  if (c.A >= (int64_t)kPairRowsPerExpert * c.E)
    return from_cuda(launch_ffn_tc2(c, xperm, expert_start, kept_counts, w_gate_up, w_down, xs,
                                    shared_gate_up, shared_down, yperm, yshared, h, status, s));
  return from_cuda(launch_ffn_tc(c, xperm, expert_start, kept_counts, w_gate_up, w_down, xs,
                                 shared_gate_up, shared_down, yperm, yshared, h, status, s));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_send_rows(const moe_config* cfg, int64_t* rows) {
  Cfg c;
  const moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!rows) return MOE_ERR_INVALID_ARG;
  *rows = c.send_rows;
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  Cfg c;
  const moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = layout(c).total;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* w_router,
                     const float* b_router, const float* sel_bias, float* logits,
                     int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                     void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!x || !w_router || !logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(logits, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_w, 4) || (b_router && !aligned(b_router, 4)) ||
      (sel_bias && !aligned(sel_bias, 4)))
    return MOE_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = ws_check(c, workspace, workspace_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  char* ws = static_cast<char*>(workspace);
  return from_cuda(launch_route(c, x, w_router, b_router, sel_bias, logits, topk_idx, topk_w,
                                ws + w.router_w, reinterpret_cast<float*>(ws + w.router_partial),
                                reinterpret_cast<int*>(ws + w.status),
                                static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x, void* xperm,
                        int32_t* expert_counts, int32_t* kept_counts, int32_t* expert_start,
                        int32_t* rank_counts, int32_t* rank_offsets, int32_t* slot_of,
                        int32_t* perm_src, int32_t* num_kept, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!topk_idx || !expert_counts || !kept_counts || !expert_start || !rank_counts ||
      !rank_offsets || !slot_of || !perm_src || !num_kept)
    return MOE_ERR_INVALID_ARG;
  if (xperm && (!x || !aligned(x, 16) || !aligned(xperm, 16))) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {topk_idx, expert_counts, kept_counts, expert_start, rank_counts,
                        rank_offsets, slot_of, perm_src, num_kept};
  for (const void* p : ints)
    if (!aligned(p, 4)) return MOE_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = ws_check(c, workspace, workspace_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + w.chunk_hist);
  return from_cuda(launch_dispatch(c, topk_idx, x, xperm, expert_counts, kept_counts, expert_start,
                                   rank_counts, rank_offsets, slot_of, perm_src, num_kept, hist,
                                   static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                                void* xperm, int32_t* expert_counts, int32_t* kept_counts,
                                int32_t* expert_start, int32_t* rank_counts,
                                int32_t* rank_offsets, int32_t* slot_of, int32_t* perm_src,
                                int32_t* num_kept, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!topk_idx || !expert_counts || !kept_counts || !expert_start || !rank_counts ||
      !rank_offsets || !slot_of || !perm_src || !num_kept)
    return MOE_ERR_INVALID_ARG;
  if (xperm && (!x || !aligned(x, 16) || !aligned(xperm, 16))) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {topk_idx, expert_counts, kept_counts, expert_start, rank_counts,
                        rank_offsets, slot_of, perm_src, num_kept};
  for (const void* p : ints)
    if (!aligned(p, 4)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)c.n_chunks * c.E > kNoAllocHistInts) return MOE_ERR_WORKSPACE;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_dispatch_noalloc(c, topk_idx, x, xperm, expert_counts, kept_counts,
                                           expert_start, rank_counts, rank_offsets, slot_of,
                                           perm_src, num_kept, static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* xperm, const int32_t* expert_start,
                          const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                          const void* x, const void* shared_gate_up, const void* shared_down,
                          void* yperm, void* yshared, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return expert_ffn_impl(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                         shared_gate_up, shared_down, yperm, yshared, workspace, workspace_bytes,
                         stream, -1);
}

moe_status moe_selftest_ffn_stall(const moe_config* cfg, const void* xperm,
                                  const int32_t* expert_start, const int32_t* kept_counts,
                                  const void* w_gate_up, const void* w_down, const void* x,
                                  const void* shared_gate_up, const void* shared_down, void* yperm,
                                  void* yshared, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  return expert_ffn_impl(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                         shared_gate_up, shared_down, yperm, yshared, workspace, workspace_bytes,
                         stream, 0);
}

moe_status moe_saved_size(const moe_config* cfg, size_t* bytes) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = saved_bytes(c);
  return MOE_OK;
}

moe_status moe_expert_ffn_save(const moe_config* cfg, const void* xperm,
                               const int32_t* expert_start, const int32_t* kept_counts,
                               const void* w_gate_up, const void* w_down, const void* x,
                               const void* shared_gate_up, const void* shared_down, void* yperm,
                               void* yshared, void* saved, size_t saved_size, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!saved) return MOE_ERR_INVALID_ARG;
  return expert_ffn_impl(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                         shared_gate_up, shared_down, yperm, yshared, workspace, workspace_bytes,
                         stream, -1, saved, saved_size);
}

moe_status moe_combine(const moe_config* cfg, const void* yperm, const int32_t* slot_of,
                       const float* topk_w, const void* residual, const void* yshared, void* out,
                       void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!yperm || !slot_of || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(yperm, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16)) ||
      (yshared && !aligned(yshared, 16)) || !aligned(slot_of, 4) || !aligned(topk_w, 4))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_combine(c, yperm, slot_of, topk_w, residual, yshared, out,
                                  static_cast<cudaStream_t>(stream)));
}

moe_status moe_bias_update(const moe_config* cfg, const int32_t* expert_counts, float* sel_bias,
                           float step, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!expert_counts || !sel_bias || !aligned(expert_counts, 4) || !aligned(sel_bias, 4))
    return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(step)) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_bias_update(c, expert_counts, sel_bias, step,
                                      static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_q8(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                           int8_t* xperm_q, float* xscale, int32_t* expert_counts,
                           int32_t* kept_counts, int32_t* expert_start, int32_t* rank_counts,
                           int32_t* rank_offsets, int32_t* slot_of, int32_t* perm_src,
                           int32_t* num_kept, void* workspace, size_t workspace_bytes,
                           void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!topk_idx || !x || !xperm_q || !xscale || !expert_counts || !kept_counts ||
      !expert_start || !rank_counts || !rank_offsets || !slot_of || !perm_src || !num_kept)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xperm_q, 16)) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {topk_idx, xscale, expert_counts, kept_counts, expert_start, rank_counts,
                        rank_offsets, slot_of, perm_src, num_kept};
  for (const void* p : ints)
    if (!aligned(p, 4)) return MOE_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = ws_check(c, workspace, workspace_bytes, &w)) != MOE_OK) return st;
  if ((st = check_device()) != MOE_OK) return st;
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + w.chunk_hist);
  return from_cuda(launch_dispatch_q8(c, topk_idx, x, xperm_q, xscale, expert_counts, kept_counts,
                                      expert_start, rank_counts, rank_offsets, slot_of, perm_src,
                                      num_kept, hist, static_cast<cudaStream_t>(stream)));
}

moe_status moe_quant_rows(const moe_config* cfg, const void* rows, const int32_t* perm_src,
                          int8_t* q, float* scale, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!rows || !perm_src || !q || !scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(rows, 16) || !aligned(q, 16) || !aligned(perm_src, 4) || !aligned(scale, 4))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_quant_rows(c, rows, perm_src, q, scale,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status moe_dequant_rows(const moe_config* cfg, const int8_t* q, const float* scale,
                            const int32_t* perm_src, void* rows, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!rows || !perm_src || !q || !scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(rows, 16) || !aligned(q, 16) || !aligned(perm_src, 4) || !aligned(scale, 4))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_dequant_rows(c, q, scale, perm_src, rows,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_q8(const moe_config* cfg, const int8_t* yperm_q, const float* yscale,
                          const int32_t* slot_of, const float* topk_w, const void* residual,
                          const void* yshared, void* out, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!yperm_q || !yscale || !slot_of || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(yperm_q, 16) || !aligned(out, 16) || !aligned(yscale, 4) || !aligned(slot_of, 4) ||
      !aligned(topk_w, 4))
    return MOE_ERR_INVALID_ARG;
  if ((residual && !aligned(residual, 16)) || (yshared && !aligned(yshared, 16)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_combine_q8(c, yperm_q, yscale, slot_of, topk_w, residual, yshared, out,
                                     static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- backward
moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const size_t ffn = ffn_backward_ws_bytes(c), router = router_bwd_ws_bytes(c);
  *bytes = 256 + round_up(ffn > router ? ffn : router);
  return MOE_OK;
}

moe_status moe_combine_backward(const moe_config* cfg, const void* dout, const void* yperm,
                                const int32_t* slot_of, const float* topk_w, void* dyperm,
                                float* dtopk_w, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!dout || !yperm || !slot_of || !topk_w || !dyperm || !dtopk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(dout, 16) || !aligned(yperm, 16) || !aligned(dyperm, 16) || !aligned(slot_of, 4) ||
      !aligned(topk_w, 4) || !aligned(dtopk_w, 4))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_combine_backward(c, dout, yperm, slot_of, topk_w, dyperm, dtopk_w,
                                           static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn_backward(const moe_config* cfg, const void* xperm,
                                   const int32_t* expert_start, const int32_t* kept_counts,
                                   const void* w_gate_up, const void* w_down, const void* x,
                                   const void* shared_gate_up, const void* shared_down,
                                   const void* dyperm, const void* dout, void* dxperm,
                                   void* dx_shared, void* dw_gate_up, void* dw_down,
                                   void* dshared_gate_up, void* dshared_down, const void* saved,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (c.act != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  const void* req[] = {xperm, w_gate_up, w_down, dyperm, dxperm, dw_gate_up, dw_down};
  for (const void* q : req)
    if (!q || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  if (!expert_start || !kept_counts || !aligned(expert_start, 4) || !aligned(kept_counts, 4))
    return MOE_ERR_INVALID_ARG;
  if (c.Fs > 0) {
    const void* sh[] = {x, shared_gate_up, shared_down, dout, dx_shared, dshared_gate_up,
                        dshared_down};
    for (const void* q : sh)
      if (!q || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  }
  if (saved && !aligned(saved, 16)) return MOE_ERR_INVALID_ARG;
  size_t need = 0;
  if ((st = moe_backward_workspace_size(cfg, &need)) != MOE_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
  if ((st = check_device()) != MOE_OK) return st;
  int* status = static_cast<int*>(workspace);
  return from_cuda(launch_ffn_backward(c, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                                       shared_gate_up, shared_down, dyperm, dout, dxperm,
                                       dx_shared, dw_gate_up, dw_down, dshared_gate_up,
                                       dshared_down, saved, static_cast<char*>(workspace) + 256,
                                       status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_backward(const moe_config* cfg, const void* x, const float* w_router,
                              const float* logits, const int32_t* topk_idx, const float* dtopk_w,
                              float* dlogits, float* dx_router, float* dw_router,
                              float* db_router, void* workspace, size_t workspace_bytes,
                              void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!logits || !topk_idx || !dtopk_w || !dlogits) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(dtopk_w, 4) || !aligned(dlogits, 4))
    return MOE_ERR_INVALID_ARG;
  if (dx_router && (!w_router || !aligned(w_router, 16) || !aligned(dx_router, 16)))
    return MOE_ERR_INVALID_ARG;
  if ((dw_router == nullptr) != (db_router == nullptr)) return MOE_ERR_INVALID_ARG;
  if (dw_router && (!x || !aligned(x, 16) || !aligned(dw_router, 16) || !aligned(db_router, 4)))
    return MOE_ERR_INVALID_ARG;
  void* ws = nullptr;
  int* status = nullptr;
  if (dw_router) {
    size_t need = 0;
    if ((st = moe_backward_workspace_size(cfg, &need)) != MOE_OK) return st;
    if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
    status = static_cast<int*>(workspace);
    ws = static_cast<char*>(workspace) + 256;
  }
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_route_backward(c, x, w_router, logits, topk_idx, dtopk_w, dlogits,
                                         dx_router, dw_router, db_router, ws, status,
                                         static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_backward(const moe_config* cfg, const void* dxperm, const int32_t* slot_of,
                                 const void* dout, const void* dx_shared, const float* dx_router,
                                 void* dx, void* stream) {
  Cfg c;
  moe_status st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  if (!dxperm || !slot_of || !dout || !dx) return MOE_ERR_INVALID_ARG;
  if (!aligned(dxperm, 16) || !aligned(dout, 16) || !aligned(dx, 16) || !aligned(slot_of, 4) ||
      (dx_shared && !aligned(dx_shared, 16)) || (dx_router && !aligned(dx_router, 16)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return from_cuda(launch_dispatch_backward(c, dxperm, slot_of, dout, dx_shared, dx_router, dx,
                                            static_cast<cudaStream_t>(stream)));
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK: success";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid size, pointer or alignment";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: device is not compute capability 10.3";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than moe_workspace_size";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA launch or runtime call failed";
  }
  return "unknown moe_status";
}

}  // extern "C"
