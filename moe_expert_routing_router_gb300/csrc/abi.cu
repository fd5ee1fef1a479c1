// Host side of the C ABI declared in include/moe_router.h: argument checks,
// workspace layout, choice of the kernel variant, grid sizing and launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <unordered_map>

#include "moe_router.h"
#include "router_ext.cuh"
#include "router_kernels.cuh"
#include "router_table.h"
#include "sinkhorn.h"
#include "eplb.h"
#include "taot_match.h"

namespace {

using moe::RouterParams;
using moe::RouterVariant;

constexpr int kGridMax = moe::kGridMax;              // CTAs of the persistent kernel
constexpr size_t kAlign = 256;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;   // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<unsigned long long*> g_trace{nullptr};
std::atomic<unsigned> g_barrier_extra{0};
std::atomic<int> g_trace_ctas{0};

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace: [Ctrl][group_hist][pfix][tile_hist E x kGridMax][P_part E x kGridMax][counts E].
// The group sums must be zero when a launch starts, so they have a region of
// their own at a fixed place and of a fixed size, whatever E: calls with
// different E on one workspace never write into it with anything but sums
// that their own CTA 0 clears again.
struct WsLayout {
  size_t ctrl = 0, group_hist = 0, pfix = 0, tile_hist = 0, p_part = 0, counts = 0, total = 0;
};

constexpr size_t kGroupHistBytes = size_t(moe::kGroupMax) * MOE_MAX_EXPERTS * sizeof(int32_t);
// A split fused step's sums of p in fixed point: two 64-bit integers per
// expert, zero between launches like the group sums (so both sit before
// tile_hist, in the part moe_get_device_status clears after a failure).
constexpr size_t kPfixBytes = size_t(2) * moe::kMaxExperts * sizeof(unsigned long long);
static_assert(moe::kMaxExperts == MOE_MAX_EXPERTS, "expert limit");

WsLayout ws_layout(int E) {
  WsLayout w;
  w.ctrl = 0;
  w.group_hist = align_up(sizeof(moe::Ctrl));
  w.pfix = w.group_hist + align_up(kGroupHistBytes);
  w.tile_hist = w.pfix + align_up(kPfixBytes);
  w.p_part = w.tile_hist + align_up(size_t(E) * kGridMax * sizeof(int32_t));
  w.counts = w.p_part + align_up(size_t(E) * kGridMax * sizeof(float));
  w.total = w.counts + align_up(size_t(E) * sizeof(int32_t));
  return w;
}

// Device address of the fixed scratch array of moe_router_step_static on the
// current device (defined with that entry point at the end of this file).
moe_status static_scratch(void** out);

// Per-device, per-kernel occupancy (blocks per SM) and SM count.
struct DeviceInfo {
  int sms = 0;
};

std::mutex g_mu;
std::unordered_map<int, DeviceInfo> g_devices;
std::unordered_map<std::string, int> g_occupancy;

moe_status device_info(DeviceInfo* out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceInfo d;
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    it = g_devices.emplace(dev, d).first;
  }
  *out = it->second;
  *dev_out = dev;
  return MOE_OK;
}

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `smem` (never lowers it), with one driver call per device, kernel and
// larger size.
moe_status raise_smem_limit(const void* func, size_t smem) {
  if (smem <= 48 * 1024) return MOE_OK;
  int dev = 0;
  cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return cuda_fail(ge, "cudaGetDevice");
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> raised;
  std::lock_guard<std::mutex> lk(mu);
  size_t& have = raised[{dev, func}];
  if (have < smem) {
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    have = smem;
  }
  return MOE_OK;
}

moe_status occupancy(const void* func, int threads, size_t smem, int dev, int* blocks) {
  char key[96];
  snprintf(key, sizeof(key), "%d:%p:%d:%zu", dev, func, threads, smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occupancy.find(key);
    if (it != g_occupancy.end()) {
      *blocks = it->second;
      return MOE_OK;
    }
  }
  moe_status s = raise_smem_limit(func, smem);
  if (s != MOE_OK) return s;
  int b = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, func, threads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (b < 1) return fail(MOE_ERR_CUDA, "kernel does not fit on an SM (smem %zu bytes)", smem);
  std::lock_guard<std::mutex> lk(g_mu);
  g_occupancy[key] = b;
  *blocks = b;
  return MOE_OK;
}

// Picks the compiled variant for (dtype, E): a staged variant (rows streamed
// through the shared-memory ring) with the smallest coverage when a row is a
// multiple of 16 bytes and the arrays are 16-byte aligned, else the smallest
// direct variant (one element per load, any E).
const RouterVariant* pick_variant(moe_dtype dt, int E, bool aligned16) {
  const int esize = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const bool staged_ok = aligned16 && (E * esize) % 16 == 0;
  int ns = 0, nd = 0;
  const RouterVariant* st = dt == MOE_DTYPE_BF16 ? moe::router_variants_bf16_staged(&ns) : moe::router_variants_fp32_staged(&ns);
  const RouterVariant* di = dt == MOE_DTYPE_BF16 ? moe::router_variants_bf16_direct(&nd) : moe::router_variants_fp32_direct(&nd);
  const RouterVariant* best = nullptr;
  auto cover = [](const RouterVariant* v) { return v->LPR * v->VW * v->NV; };
  if (staged_ok)
    for (int i = 0; i < ns; ++i)
      if (cover(&st[i]) >= E && E % st[i].VW == 0 && (!best || cover(&st[i]) < cover(best))) best = &st[i];
  if (!best)
    for (int i = 0; i < nd; ++i)
      if (cover(&di[i]) >= E && (!best || cover(&di[i]) < cover(best))) best = &di[i];
  return best;
}

// The extended step's kernels of a plain variant (the same row layout), or null.
const moe::StepExtVariant* step_ext_variant(moe_dtype dt, const RouterVariant* v) {
  int n = 0;
  const moe::StepExtVariant* t =
      dt == MOE_DTYPE_BF16 ? (v->staged ? moe::step_ext_bf16_staged(&n) : moe::step_ext_bf16_direct(&n))
                           : (v->staged ? moe::step_ext_fp32_staged(&n) : moe::step_ext_fp32_direct(&n));
  for (int i = 0; i < n; ++i)
    if (t[i].LPR == v->LPR && t[i].VW == v->VW && t[i].NV == v->NV && t[i].NR == v->NR &&
        t[i].min_blocks == v->min_blocks)
      return &t[i];
  return nullptr;
}

moe_status check_router_args(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k) {
  if (dt != MOE_DTYPE_FP32 && dt != MOE_DTYPE_BF16) return fail(MOE_ERR_UNSUPPORTED, "dtype %d is not fp32 (0) or bf16 (1)", int(dt));
  if (!logits) return fail(MOE_ERR_INVALID, "logits is NULL");
  if (T < 1 || T >= (int64_t(1) << 31)) return fail(MOE_ERR_INVALID, "T = %lld outside [1, 2^31)", (long long)T);
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_INVALID, "E = %d outside [1, %d]", E, MOE_MAX_EXPERTS);
  if (k < 1 || k > MOE_MAX_TOPK || k > E) return fail(MOE_ERR_INVALID, "k = %d outside [1, min(E, %d)]", k, MOE_MAX_TOPK);
  if (T * (int64_t)k >= (int64_t(1) << 31)) return fail(MOE_ERR_INVALID, "T*k = %lld does not fit int32", (long long)(T * k));
  if (!aligned(logits, dt == MOE_DTYPE_BF16 ? 2 : 4)) return fail(MOE_ERR_INVALID, "logits is not element aligned");
  return MOE_OK;
}

moe_status check_ws(void* ws, size_t ws_bytes, int E) {
  if (!ws) return fail(MOE_ERR_INVALID, "workspace is NULL");
  if (!aligned(ws, kAlign)) return fail(MOE_ERR_INVALID, "workspace is not 256-byte aligned");
  const size_t need = ws_layout(E).total;
  if (ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return MOE_OK;
}

void bind_ws(RouterParams& p, void* ws, int E) {
  const WsLayout w = ws_layout(E);
  char* base = static_cast<char*>(ws);
  p.ctrl = reinterpret_cast<moe::Ctrl*>(base + w.ctrl);
  p.tile_hist = reinterpret_cast<int32_t*>(base + w.tile_hist);
  p.group_hist = reinterpret_cast<int32_t*>(base + w.group_hist);
  p.pfix = reinterpret_cast<unsigned long long*>(base + w.pfix);
  p.P_part = reinterpret_cast<float*>(base + w.p_part);
  p.counts_ws = reinterpret_cast<int32_t*>(base + w.counts);
  p.G_stride = kGridMax;
  p.timeout_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.trace = g_trace.load(std::memory_order_relaxed);
  p.barrier_extra = g_barrier_extra.load(std::memory_order_relaxed);
}

int64_t capacity_of(int64_t T, int32_t E, int32_t k, double cf) {
  const int64_t per_expert = (T * k + E - 1) / E;
  return (int64_t)std::ceil(double(per_expert) * cf);
}

// Launch geometry of the persistent kernel: every CTA resident (cooperative
// launch), at least one row group per consumer warp, at most kGridMax CTAs;
// for staged variants, ring stages of about 16 KB and as many slots as fit in
// the shared memory left per CTA (or as the chunk needs).
struct Geometry {
  int G = 1, rows_per_stage = 0, n_slots = 0, asg_cap = 0, rstat_cap = 0;
  size_t smem = 0;
};

constexpr size_t kSmemPerSm = 228 * 1024;      // GB300 shared memory per SM
constexpr size_t kSmemReservedPerCta = 1024;
constexpr int kStageBytes = 65536;             // target size of one ring stage (several rows per consumer warp)
constexpr int kMaxAsgSmem = 12288;             // assignments per CTA kept in shared memory for the dispatch
constexpr int kMaxRowStats = 4096;             // rows per CTA whose softmax statistics stay in shared memory

// fused: the launch runs the fused step (forward, dispatch and backward), whose
// CTAs keep their dispatch and the rows' softmax statistics in shared memory
// when these fit beside at least two ring slots.
// ext: the extended step's kernel of the variant (its pick slots hold 32-bit
// selection keys and its occupancy sets the grid), or null for the plain kernels.
moe_status persistent_geometry(const RouterVariant* v, moe_dtype dt, int64_t T, int E, int k, bool fused,
                               Geometry* out, const void* ext = nullptr) {
  DeviceInfo d;
  int dev = 0;
  moe_status s = device_info(&d, &dev);
  if (s != MOE_OK) return s;
  const int esize = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const int kb = ext != nullptr ? int(sizeof(uint32_t))
                 : dt == MOE_DTYPE_BF16 ? int(sizeof(moe::Bf16::Key)) : int(sizeof(moe::Fp32::Key));
  const int group_rows = moe::kConsumerWarps * (moe::kWarp / v->LPR) * v->NR;
  Geometry g;
  const size_t fixed = moe::router_smem_layout(E, kb, 0, 0).total;
  const size_t budget = kSmemPerSm / size_t(v->min_blocks) - kSmemReservedPerCta;
  size_t stage_bytes = 0;
  if (v->staged) {
    const int row_bytes = E * esize;
    g.rows_per_stage = std::max(group_rows, (kStageBytes / row_bytes) / group_rows * group_rows);
    stage_bytes = size_t(g.rows_per_stage) * row_bytes;
    g.n_slots = int(std::max<size_t>(1, std::min<size_t>(moe::kMaxSlots, (budget - fixed) / stage_bytes)));
  }
  size_t smem = moe::router_smem_layout(E, kb, g.n_slots, int(stage_bytes)).total;
  int bf = 0, bs = 0;
  if (ext != nullptr) {
    if ((s = occupancy(ext, moe::kThreads, smem, dev, &bs)) != MOE_OK) return s;
    bf = bs;
  } else {
    if ((s = occupancy(v->fwd, moe::kThreads, smem, dev, &bf)) != MOE_OK) return s;
    if ((s = occupancy(v->step, moe::kThreads, smem, dev, &bs)) != MOE_OK) return s;
  }
  if (ext == nullptr && v->step_split != nullptr) {
    int bss = 0;
    if ((s = occupancy(v->step_split, moe::kThreads, smem, dev, &bss)) != MOE_OK) return s;
    bs = std::min(bs, bss);
  }
  const int64_t cap = std::min<int64_t>(int64_t(std::min(bf, bs)) * d.sms, kGridMax);
  const int64_t want = (T + group_rows - 1) / group_rows;
  g.G = int(std::max<int64_t>(1, std::min(cap, want)));
  if (v->staged) {
    const int64_t chunk = (T + g.G - 1) / g.G;
    if (fused) {
      const int64_t rows = (chunk + 15) / 16 * 16;
      if (rows <= kMaxRowStats &&
          moe::router_smem_layout(E, kb, 0, 0, 0, int(rows)).total + 2 * stage_bytes <= budget)
        g.rstat_cap = int(rows);
      const int64_t asg = (chunk * k + 7) / 8 * 8;
      if (asg <= kMaxAsgSmem &&
          moe::router_smem_layout(E, kb, 0, 0, int(asg), g.rstat_cap).total + 2 * stage_bytes <= budget)
        g.asg_cap = int(asg);
      const size_t with = moe::router_smem_layout(E, kb, 0, 0, g.asg_cap, g.rstat_cap).total;
      g.n_slots = int(std::max<size_t>(1, std::min<size_t>(moe::kMaxSlots, (budget - with) / stage_bytes)));
    }
    const int64_t stages = (chunk + g.rows_per_stage - 1) / g.rows_per_stage;   // no more slots than stages
    g.n_slots = int(std::max<int64_t>(1, std::min<int64_t>(g.n_slots, stages)));
    smem = moe::router_smem_layout(E, kb, g.n_slots, int(stage_bytes), g.asg_cap, g.rstat_cap).total;
  }
  g.smem = smem;
  *out = g;
  return MOE_OK;
}

moe_status launch_persistent(const void* func, const RouterParams& p, size_t smem, cudaStream_t stream) {
  if (p.trace != nullptr && p.G > g_trace_ctas.load(std::memory_order_relaxed))
    return fail(MOE_ERR_INVALID, "trace buffer holds %d CTAs, the launch has %d", g_trace_ctas.load(), p.G);
  {
    moe_status s = raise_smem_limit(func, smem);
    if (s != MOE_OK) return s;
  }
  // Cooperative (every CTA resident: the grid barrier) and, where the driver
  // takes it, with programmatic dependent launch: the launch may be scheduled
  // while the previous kernel of the stream finishes, and waits for it in the
  // kernel's prologue (griddepcontrol.wait) before touching memory.
  static std::atomic<int> pdl_ok{1};
  if (pdl_ok.load(std::memory_order_relaxed)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.G);
    cfg.blockDim = dim3(moe::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeCooperative;
    attrs[0].val.cooperative = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    void* args[] = {const_cast<RouterParams*>(&p)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
    if (e == cudaSuccess) return MOE_OK;
    (void)cudaGetLastError();                 // not taken: fall back to the plain cooperative launch
    pdl_ok.store(0, std::memory_order_relaxed);
  }
  void* args[] = {const_cast<RouterParams*>(&p)};
  cudaError_t e = cudaLaunchCooperativeKernel(func, dim3(p.G), dim3(moe::kThreads), args, smem, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
  return MOE_OK;
}

RouterParams base_params(const void* logits, int64_t T, int32_t E, int32_t k) {
  RouterParams p;
  std::memset(&p, 0, sizeof(p));
  p.logits = logits;
  p.T = T;
  p.E = E;
  p.k = k;
  return p;
}

moe_status check_fwd_outputs(int32_t k, float alpha, int32_t renorm, int32_t n_ranks, int32_t E,
                             const void* idx, const void* gate, const void* counts, const void* f,
                             const void* P, const void* scalars, const void* rank_load) {
  if (!(alpha >= 0.f) || !std::isfinite(alpha)) return fail(MOE_ERR_INVALID, "alpha must be finite and >= 0");
  if (renorm < -1 || renorm > 1) return fail(MOE_ERR_INVALID, "renorm must be -1, 0 or 1");
  if (n_ranks < 0 || n_ranks > MOE_MAX_RANKS || (n_ranks > 0 && E % n_ranks != 0))
    return fail(MOE_ERR_INVALID, "n_ranks = %d must be 0 or a divisor of E in [1, %d]", n_ranks, MOE_MAX_RANKS);
  if (!idx || !gate || !counts || !f || !P || !scalars) return fail(MOE_ERR_INVALID, "a forward output is NULL");
  if (n_ranks > 0 && !rank_load) return fail(MOE_ERR_INVALID, "rank_load is NULL with n_ranks > 0");
  (void)k;
  return MOE_OK;
}

// The bias-routing / masked-P forward and full-backward kernels for (dtype, E):
// the vector-load layout with the smallest coverage when rows are a multiple
// of 16 bytes and the arrays 16-byte aligned, else the one-element-per-load
// layout.
const moe::ExtVariant* pick_ext_variant(moe_dtype dt, int E, bool aligned16) {
  const int esize = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const bool vec_ok = aligned16 && (E * esize) % 16 == 0;
  int n = 0;
  const moe::ExtVariant* all = dt == MOE_DTYPE_BF16 ? moe::ext_variants_bf16(&n) : moe::ext_variants_fp32(&n);
  auto cover = [](const moe::ExtVariant* v) { return v->LPR * v->VW * v->NV; };
  const moe::ExtVariant* best = nullptr;
  for (int pass = vec_ok ? 1 : 0; pass >= 0 && !best; --pass)
    for (int i = 0; i < n; ++i)
      if (all[i].vec == pass && cover(&all[i]) >= E && E % all[i].VW == 0 && (!best || cover(&all[i]) < cover(best)))
        best = &all[i];
  return best;
}

}  // namespace

// moe_dispatch and moe_dispatch_sharded: the capacity is that of T_cap tokens
// (the whole batch), cap_base null for a batch on one rank.
static moe_status dispatch_impl(const int32_t* idx, int64_t T, int32_t E, int32_t k, double capacity_factor,
                                int64_t T_cap, const int32_t* cap_base,
                                int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                int32_t* n_dropped, int64_t* capacity_out,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!idx) return fail(MOE_ERR_INVALID, "idx is NULL");
  if (T < 1 || T >= (int64_t(1) << 31)) return fail(MOE_ERR_INVALID, "T = %lld outside [1, 2^31)", (long long)T);
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_INVALID, "E = %d outside [1, %d]", E, MOE_MAX_EXPERTS);
  if (k < 1 || k > MOE_MAX_TOPK || k > E) return fail(MOE_ERR_INVALID, "k = %d outside [1, min(E, %d)]", k, MOE_MAX_TOPK);
  if (T * (int64_t)k >= (int64_t(1) << 31)) return fail(MOE_ERR_INVALID, "T*k does not fit int32");
  if (!(capacity_factor > 0.0) || !std::isfinite(capacity_factor)) return fail(MOE_ERR_INVALID, "capacity_factor must be > 0");
  if (!perm || !slot || !offsets || !kept || !n_dropped) return fail(MOE_ERR_INVALID, "a dispatch output is NULL");
  moe_status s = check_ws(ws, ws_bytes, E);
  if (s != MOE_OK) return s;
  const int64_t C = capacity_of(T_cap, E, k, capacity_factor);
  if (capacity_out) *capacity_out = C;
  RouterParams p = base_params(nullptr, T, E, k);
  p.idx_in = idx;
  p.cap_base = cap_base;
  p.C = int(std::min<int64_t>(C, INT32_MAX));
  p.perm = perm; p.slot = slot; p.offsets = offsets; p.kept = kept; p.n_dropped = n_dropped;
  bind_ws(p, ws, E);
  DeviceInfo d;
  int dev = 0;
  if ((s = device_info(&d, &dev)) != MOE_OK) return s;
  const void* func = moe::dispatch_kernel();
  const int kb = int(sizeof(moe::Bf16::Key));                 // a bf16 instance
  size_t smem = moe::router_smem_layout(E, kb, 0, 0).total;
  int blocks = 0;
  if ((s = occupancy(func, moe::kThreads, smem, dev, &blocks)) != MOE_OK) return s;
  const int64_t cap = std::min<int64_t>(int64_t(blocks) * d.sms, kGridMax);
  const int64_t want = (T * k + 2047) / 2048;
  p.G = int(std::max<int64_t>(1, std::min(cap, want)));
  p.n_groups = (p.G + moe::kGroupCtas - 1) / moe::kGroupCtas;
  // each CTA's assignments (expert id, rank within the CTA) in shared memory when they fit
  const int64_t asg = ((T * k + p.G - 1) / p.G + 7) / 8 * 8;
  const size_t with = moe::router_smem_layout(E, kb, 0, 0, int(std::min<int64_t>(asg, INT32_MAX))).total;
  if (asg <= kMaxAsgSmem && with <= kSmemPerSm - kSmemReservedPerCta) {
    p.asg_cap = int(asg);
    smem = with;
  }
  return launch_persistent(func, p, smem, stream);
}


extern "C" {

size_t moe_router_workspace_size(int64_t T, int32_t E, int32_t k) {
  if (T < 1 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_TOPK || k > E) return 0;
  return ws_layout(E).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || !aligned(ws, kAlign)) return fail(MOE_ERR_INVALID, "workspace is NULL or not 256-byte aligned");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return MOE_OK;
}

moe_status moe_get_device_status(void* ws, moe_stream_t stream, int32_t* flags) {
  if (!flags) return fail(MOE_ERR_INVALID, "NULL argument");
  if (!ws) {                       // the fixed scratch of moe_router_step_static on this device
    moe_status s = static_scratch(&ws);
    if (s != MOE_OK) return s;
  }
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  moe::Ctrl c{};
  e = cudaMemcpy(&c, ws, sizeof(moe::Ctrl), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  const int32_t v = int32_t(c.sync >> 32);
  *flags = v;
  if (v != 0) {
    // Clear the flags, the barrier state and the failed launch's group sums
    // for the next call.
    e = cudaMemset(ws, 0, ws_layout(1).tile_hist);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
    return fail(MOE_ERR_TIMEOUT, "device wait expired (flags 0x%x)", unsigned(v));
  }
  return MOE_OK;
}

int64_t moe_dispatch_capacity(int64_t T, int32_t E, int32_t k, double capacity_factor) {
  if (T < 1 || T >= (int64_t(1) << 40) || E < 1 || k < 1 || !(capacity_factor > 0.0) || !std::isfinite(capacity_factor)) return -1;
  return capacity_of(T, E, k, capacity_factor);
}

moe_status moe_router_fwd(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                          float alpha, int32_t renorm, int32_t n_ranks,
                          int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                          float* scalars, int32_t* rank_load,
                          void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_router_args(logits, dt, T, E, k);
  if (s != MOE_OK) return s;
  if ((s = check_fwd_outputs(k, alpha, renorm, n_ranks, E, idx, gate, counts, f, P, scalars, rank_load)) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, E)) != MOE_OK) return s;
  const RouterVariant* v = pick_variant(dt, E, aligned(logits, 16));
  if (!v) return fail(MOE_ERR_INVALID, "no kernel variant for E = %d", E);
  RouterParams p = base_params(logits, T, E, k);
  p.alpha = alpha;
  p.renorm = renorm < 0 ? (k > 1) : renorm;
  p.n_ranks = n_ranks;
  p.idx = idx; p.gate = gate; p.counts = counts; p.f = f; p.P = P; p.scalars = scalars; p.rank_load = rank_load;
  bind_ws(p, ws, E);
  Geometry geo;
  if ((s = persistent_geometry(v, dt, T, E, k, false, &geo)) != MOE_OK) return s;
  p.G = geo.G;
  p.n_groups = (p.G + moe::kGroupCtas - 1) / moe::kGroupCtas;
  p.rows_per_stage = geo.rows_per_stage;
  p.n_slots = geo.n_slots;
  p.asg_cap = geo.asg_cap;
  p.rstat_cap = geo.rstat_cap;
  return launch_persistent(v->fwd, p, geo.smem, stream);
}

moe_status moe_router_bwd(const void* logits, moe_dtype dt, int64_t T, int32_t E, float alpha,
                          const float* f, float grad_scale, float* dlogits, moe_stream_t stream) {
  moe_status s = check_router_args(logits, dt, T, E, 1);
  if (s != MOE_OK) return s;
  if (!(alpha >= 0.f) || !std::isfinite(alpha)) return fail(MOE_ERR_INVALID, "alpha must be finite and >= 0");
  if (!std::isfinite(grad_scale)) return fail(MOE_ERR_INVALID, "grad_scale must be finite");
  if (!f || !dlogits) return fail(MOE_ERR_INVALID, "f or dlogits is NULL");
  if (!aligned(dlogits, 4) || !aligned(f, 4)) return fail(MOE_ERR_INVALID, "f or dlogits is not 4-byte aligned");
  const RouterVariant* v = pick_variant(dt, E, aligned(logits, 16) && aligned(dlogits, 16));
  if (!v) return fail(MOE_ERR_INVALID, "no kernel variant for E = %d", E);
  DeviceInfo d;
  int dev = 0;
  if ((s = device_info(&d, &dev)) != MOE_OK) return s;
  constexpr int kBwdThreads = 256;
  int blocks = 0;
  if ((s = occupancy(v->bwd, kBwdThreads, 0, dev, &blocks)) != MOE_OK) return s;
  const int64_t rows_per_block = int64_t(kBwdThreads / moe::kWarp) * (moe::kWarp / v->LPR);
  const int64_t want = (T + rows_per_block - 1) / rows_per_block;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(blocks) * d.sms)));
  moe::BwdParams p;
  p.logits = logits;
  p.T = T;
  p.E = E;
  p.f = f;
  p.coef = grad_scale * alpha * float(E) / float(T);
  p.dlogits = dlogits;
  void* args[] = {&p};
  cudaError_t e = cudaLaunchKernel(v->bwd, dim3(grid), dim3(kBwdThreads), args, 0, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernel");
  return MOE_OK;
}

moe_status moe_dispatch(const int32_t* idx, int64_t T, int32_t E, int32_t k, double capacity_factor,
                        int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                        int32_t* n_dropped, int64_t* capacity_out,
                        void* ws, size_t ws_bytes, moe_stream_t stream) {
  return dispatch_impl(idx, T, E, k, capacity_factor, T, nullptr, perm, slot, offsets, kept, n_dropped, capacity_out,
                       ws, ws_bytes, stream);
}

moe_status moe_dispatch_sharded(const int32_t* idx, int64_t T, int32_t E, int32_t k, double capacity_factor,
                                int64_t T_total, const int32_t* cap_base,
                                int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                int32_t* n_dropped, int64_t* capacity_out,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!cap_base) return fail(MOE_ERR_INVALID, "cap_base is NULL");
  if (!aligned(cap_base, 4)) return fail(MOE_ERR_INVALID, "cap_base is not 4-byte aligned");
  if (T_total < T) return fail(MOE_ERR_INVALID, "T_total = %lld is below this rank's T = %lld", (long long)T_total, (long long)T);
  if (k >= 1 && T_total * (int64_t)k >= (int64_t(1) << 31)) return fail(MOE_ERR_INVALID, "T_total*k does not fit int32");
  return dispatch_impl(idx, T, E, k, capacity_factor, T_total, cap_base, perm, slot, offsets, kept, n_dropped,
                       capacity_out, ws, ws_bytes, stream);
}

moe_status moe_shard_capacity_base(const int32_t* counts, int32_t G, int32_t E, int32_t rank, int32_t* cap_base,
                                   moe_stream_t stream) {
  if (!counts || !cap_base) return fail(MOE_ERR_INVALID, "counts or cap_base is NULL");
  if (G < 1 || G > moe::kMaxShards) return fail(MOE_ERR_INVALID, "G = %d outside [1, %d]", G, moe::kMaxShards);
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_INVALID, "E = %d outside [1, %d]", E, MOE_MAX_EXPERTS);
  if (rank < 0 || rank >= G) return fail(MOE_ERR_INVALID, "rank = %d outside [0, %d)", rank, G);
  if (!aligned(counts, 4) || !aligned(cap_base, 4)) return fail(MOE_ERR_INVALID, "counts or cap_base is not 4-byte aligned");
  cudaError_t e = moe::launch_shard_capacity_base(counts, G, E, rank, cap_base, stream);
  if (e != cudaSuccess) return cuda_fail(e, "shard_capacity_base launch");
  return MOE_OK;
}

}  // extern "C"

namespace {

// Every check of the fused step's arguments except the workspace's.
moe_status check_step_args(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k, float alpha,
                           int32_t renorm, int32_t n_ranks, double capacity_factor, float grad_scale,
                           int32_t* idx, float* gate, int32_t* counts, float* f, float* P, float* scalars,
                           int32_t* rank_load, int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                           int32_t* n_dropped, float* dlogits) {
  moe_status s = check_router_args(logits, dt, T, E, k);
  if (s != MOE_OK) return s;
  if ((s = check_fwd_outputs(k, alpha, renorm, n_ranks, E, idx, gate, counts, f, P, scalars, rank_load)) != MOE_OK) return s;
  if (!(capacity_factor > 0.0) || !std::isfinite(capacity_factor)) return fail(MOE_ERR_INVALID, "capacity_factor must be > 0");
  if (!std::isfinite(grad_scale)) return fail(MOE_ERR_INVALID, "grad_scale must be finite");
  if (!perm || !slot || !offsets || !kept || !n_dropped || !dlogits) return fail(MOE_ERR_INVALID, "a dispatch or backward output is NULL");
  if (!aligned(dlogits, 4)) return fail(MOE_ERR_INVALID, "dlogits is not 4-byte aligned");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_router_step(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                           float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                           float grad_scale,
                           int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                           float* scalars, int32_t* rank_load,
                           int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                           int32_t* n_dropped, float* dlogits,
                           void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_step_args(logits, dt, T, E, k, alpha, renorm, n_ranks, capacity_factor, grad_scale, idx, gate,
                                 counts, f, P, scalars, rank_load, perm, slot, offsets, kept, n_dropped, dlogits);
  if (s != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, E)) != MOE_OK) return s;
  const RouterVariant* v = pick_variant(dt, E, aligned(logits, 16) && aligned(dlogits, 16));
  if (!v) return fail(MOE_ERR_INVALID, "no kernel variant for E = %d", E);
  RouterParams p = base_params(logits, T, E, k);
  p.alpha = alpha;
  p.renorm = renorm < 0 ? (k > 1) : renorm;
  p.n_ranks = n_ranks;
  p.grad_scale = grad_scale;
  p.C = int(std::min<int64_t>(capacity_of(T, E, k, capacity_factor), INT32_MAX));
  p.idx = idx; p.gate = gate; p.counts = counts; p.f = f; p.P = P; p.scalars = scalars; p.rank_load = rank_load;
  p.perm = perm; p.slot = slot; p.offsets = offsets; p.kept = kept; p.n_dropped = n_dropped;
  p.dlogits = dlogits;
  bind_ws(p, ws, E);
  Geometry geo;
  if ((s = persistent_geometry(v, dt, T, E, k, true, &geo)) != MOE_OK) return s;
  p.G = geo.G;
  p.n_groups = (p.G + moe::kGroupCtas - 1) / moe::kGroupCtas;
  p.rows_per_stage = geo.rows_per_stage;
  p.n_slots = geo.n_slots;
  p.asg_cap = geo.asg_cap;
  p.rstat_cap = geo.rstat_cap;
  // With renormalised gates the split kernel forms the softmax sums and P in
  // the backward; it keeps its per-warp sums of p in the ring's memory at the end.
  const size_t ring_bytes = size_t(geo.n_slots) * size_t(geo.rows_per_stage) * size_t(E) * (dt == MOE_DTYPE_BF16 ? 2 : 4);
  const bool split = p.renorm != 0 && v->step_split != nullptr &&
                     ring_bytes >= size_t(moe::kConsumerWarps) * size_t(E) * sizeof(float);
  return launch_persistent(split ? v->step_split : v->step, p, geo.smem, stream);
}

moe_status moe_router_step_ex(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                              float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                              float grad_scale, const float* bias, float bias_gamma, float* bias_out,
                              int32_t masked_p, const float* dgate,
                              int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                              float* scalars, int32_t* rank_load,
                              int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                              int32_t* n_dropped, float* dlogits,
                              void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_step_args(logits, dt, T, E, k, alpha, renorm, n_ranks, capacity_factor, grad_scale, idx, gate,
                                 counts, f, P, scalars, rank_load, perm, slot, offsets, kept, n_dropped, dlogits);
  if (s != MOE_OK) return s;
  if (!aligned(bias, 4) || !aligned(bias_out, 4) || !aligned(dgate, 4))
    return fail(MOE_ERR_INVALID, "bias, bias_out or dgate is not 4-byte aligned");
  if (bias_out != nullptr && !std::isfinite(bias_gamma)) return fail(MOE_ERR_INVALID, "bias_gamma must be finite");
  if ((s = check_ws(ws, ws_bytes, E)) != MOE_OK) return s;
  const RouterVariant* v = pick_variant(dt, E, aligned(logits, 16) && aligned(dlogits, 16));
  if (!v) return fail(MOE_ERR_INVALID, "no kernel variant for E = %d", E);
  const moe::StepExtVariant* xv = step_ext_variant(dt, v);
  if (!xv) return fail(MOE_ERR_INVALID, "no extended step kernel for E = %d", E);
  const void* func = xv->step_ext;
  RouterParams p = base_params(logits, T, E, k);
  p.alpha = alpha;
  p.renorm = renorm < 0 ? (k > 1) : renorm;
  p.n_ranks = n_ranks;
  p.grad_scale = grad_scale;
  p.C = int(std::min<int64_t>(capacity_of(T, E, k, capacity_factor), INT32_MAX));
  p.bias = bias;
  p.bias_gamma = bias_gamma;
  p.bias_out = bias_out;
  p.masked_p = masked_p != 0;
  p.dgate = dgate;
  p.idx = idx; p.gate = gate; p.counts = counts; p.f = f; p.P = P; p.scalars = scalars; p.rank_load = rank_load;
  p.perm = perm; p.slot = slot; p.offsets = offsets; p.kept = kept; p.n_dropped = n_dropped;
  p.dlogits = dlogits;
  bind_ws(p, ws, E);
  Geometry geo;
  if ((s = persistent_geometry(v, dt, T, E, k, true, &geo, func)) != MOE_OK) return s;
  p.G = geo.G;
  p.n_groups = (p.G + moe::kGroupCtas - 1) / moe::kGroupCtas;
  p.rows_per_stage = geo.rows_per_stage;
  p.n_slots = geo.n_slots;
  p.asg_cap = geo.asg_cap;
  p.rstat_cap = geo.rstat_cap;
  return launch_persistent(func, p, geo.smem, stream);
}

}  // extern "C"

namespace {

// Device staging layout of moe_router_step_host: the logits, then every
// output of the step, each 256-byte aligned.
struct HostStepLayout {
  size_t logits, idx, gate, counts, f, P, scalars, rank_load, perm, slot, offsets, kept, n_dropped, dlogits, total;
};

HostStepLayout host_step_layout(moe_dtype dt, int64_t T, int32_t E, int32_t k, int32_t n_ranks) {
  const size_t esize = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const size_t tk = size_t(T) * size_t(k), te = size_t(T) * size_t(E);
  HostStepLayout L;
  size_t at = 0;
  auto take = [&at](size_t bytes) { const size_t o = at; at += align_up(bytes); return o; };
  L.logits = take(te * esize);
  L.idx = take(tk * 4);
  L.gate = take(tk * 4);
  L.counts = take(size_t(E) * 4);
  L.f = take(size_t(E) * 4);
  L.P = take(size_t(E) * 4);
  L.scalars = take(size_t(moe::kNumScalars) * 4);
  L.rank_load = take(size_t(n_ranks > 0 ? n_ranks : 0) * 4);
  L.perm = take(tk * 4);
  L.slot = take(tk * 4);
  L.offsets = take(size_t(E + 1) * 4);
  L.kept = take(size_t(E) * 4);
  L.n_dropped = take(4);
  L.dlogits = take(te * 4);
  L.total = at;
  return L;
}

}  // namespace

extern "C" {

size_t moe_router_step_host_device_size(moe_dtype dt, int64_t T, int32_t E, int32_t k, int32_t n_ranks) {
  if (T < 1 || E < 1 || k < 1 || n_ranks < 0) return 0;
  return host_step_layout(dt, T, E, k, n_ranks).total;
}

moe_status moe_router_step_host(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                                float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                                float grad_scale,
                                int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                                float* scalars, int32_t* rank_load,
                                int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                int32_t* n_dropped, float* dlogits,
                                void* dev, size_t dev_bytes, void* ws, size_t ws_bytes,
                                void* kernel_after, void* kernel_done, moe_stream_t stream) {
  // The host pointers are only checked for NULL here; the device staging
  // pointers handed to the step are checked by moe_router_step itself.
  if (!logits || !idx || !gate || !counts || !f || !P || !scalars || (n_ranks > 0 && !rank_load) || !perm ||
      !slot || !offsets || !kept || !n_dropped || !dlogits)
    return fail(MOE_ERR_INVALID, "a host input or output is NULL");
  if (dt != MOE_DTYPE_BF16 && dt != MOE_DTYPE_FP32) return fail(MOE_ERR_UNSUPPORTED, "dtype %d", int(dt));
  if (T < 1 || E < 1 || k < 1 || n_ranks < 0) return fail(MOE_ERR_INVALID, "T, E, k must be >= 1 and n_ranks >= 0");
  if (!dev || !aligned(dev, kAlign)) return fail(MOE_ERR_INVALID, "device staging buffer is NULL or not 256-byte aligned");
  const HostStepLayout L = host_step_layout(dt, T, E, k, n_ranks);
  if (dev_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "device staging buffer of %zu bytes, %zu needed", dev_bytes, L.total);
  unsigned char* d = static_cast<unsigned char*>(dev);
  const size_t esize = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const size_t tk = size_t(T) * size_t(k), te = size_t(T) * size_t(E);
  cudaError_t e = cudaMemcpyAsync(d + L.logits, logits, te * esize, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (logits in)");
  if (kernel_after) {
    e = cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(kernel_after), 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  moe_status s = moe_router_step(d + L.logits, dt, T, E, k, alpha, renorm, n_ranks, capacity_factor, grad_scale,
                                 reinterpret_cast<int32_t*>(d + L.idx), reinterpret_cast<float*>(d + L.gate),
                                 reinterpret_cast<int32_t*>(d + L.counts), reinterpret_cast<float*>(d + L.f),
                                 reinterpret_cast<float*>(d + L.P), reinterpret_cast<float*>(d + L.scalars),
                                 n_ranks > 0 ? reinterpret_cast<int32_t*>(d + L.rank_load) : nullptr,
                                 reinterpret_cast<int32_t*>(d + L.perm), reinterpret_cast<int32_t*>(d + L.slot),
                                 reinterpret_cast<int32_t*>(d + L.offsets), reinterpret_cast<int32_t*>(d + L.kept),
                                 reinterpret_cast<int32_t*>(d + L.n_dropped), reinterpret_cast<float*>(d + L.dlogits),
                                 ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  if (kernel_done) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(kernel_done), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  }
  struct Back { void* dst; size_t off, bytes; };
  const Back back[] = {
      {idx, L.idx, tk * 4}, {gate, L.gate, tk * 4}, {counts, L.counts, size_t(E) * 4}, {f, L.f, size_t(E) * 4},
      {P, L.P, size_t(E) * 4}, {scalars, L.scalars, size_t(moe::kNumScalars) * 4},
      {rank_load, L.rank_load, size_t(n_ranks) * 4}, {perm, L.perm, tk * 4}, {slot, L.slot, tk * 4},
      {offsets, L.offsets, size_t(E + 1) * 4}, {kept, L.kept, size_t(E) * 4}, {n_dropped, L.n_dropped, 4},
      {dlogits, L.dlogits, te * 4}};
  for (const Back& b : back) {
    if (b.bytes == 0) continue;
    e = cudaMemcpyAsync(b.dst, d + b.off, b.bytes, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (outputs back)");
  }
  return MOE_OK;
}

moe_status taot_sinkhorn_batched(const float* loads, int32_t B, int32_t R, int32_t ranks_per_node,
                                 float lambda, float eps, int32_t iters,
                                 float* u, float* v, float* plan, int32_t* status,
                                 moe_stream_t stream) {
  if (!loads || !u || !v || !status) return fail(MOE_ERR_INVALID, "a Sinkhorn argument is NULL");
  if (B < 1) return fail(MOE_ERR_INVALID, "B = %d must be >= 1", B);
  if (R < 1 || R > MOE_MAX_RANKS) return fail(MOE_ERR_INVALID, "R = %d outside [1, %d]", R, MOE_MAX_RANKS);
  if (ranks_per_node < 1 || ranks_per_node > R || R % ranks_per_node != 0)
    return fail(MOE_ERR_INVALID, "ranks_per_node = %d must divide R = %d", ranks_per_node, R);
  if (!(lambda > 0.f) || !std::isfinite(lambda)) return fail(MOE_ERR_INVALID, "lambda must be > 0");
  if (!std::isfinite(eps)) return fail(MOE_ERR_INVALID, "eps must be finite");
  if (iters < 0) return fail(MOE_ERR_INVALID, "iters must be >= 0");
  const double e = eps > 0.f ? double(eps) : double(lambda);
  moe::SinkhornParams p;
  p.loads = loads;
  p.B = B;
  p.R = R;
  p.ranks_per_node = ranks_per_node;
  p.iters = iters;
  const double m_node = std::exp(-1.0 / e), m_cross = std::exp(-double(lambda) / e);
  p.m_node = float(m_node);
  p.m_cross = float(m_cross);
  p.c_self = float(1.0 - m_node);
  p.c_node = float(m_node - m_cross);
  p.c_all = float(m_cross);
  p.u = u;
  p.v = v;
  p.plan = plan;
  p.plan_vec4 = plan != nullptr && R % 4 == 0 && reinterpret_cast<uintptr_t>(plan) % 16 == 0 ? 1 : 0;
  p.status = status;
  cudaError_t err = moe::launch_taot_sinkhorn(p, stream);
  if (err != cudaSuccess) return cuda_fail(err, "taot_sinkhorn launch");
  return MOE_OK;
}

moe_status moe_eplb_plan(const int32_t* loads, int32_t B, int32_t E, int32_t num_phys,
                         int32_t num_gpus, int32_t num_nodes, int32_t num_groups,
                         int32_t* phy2log, int32_t* log_count, float* gpu_load, moe_stream_t stream) {
  if (!loads || !phy2log || !log_count || !gpu_load) return fail(MOE_ERR_INVALID, "an EPLB argument is NULL");
  if (B < 1) return fail(MOE_ERR_INVALID, "B = %d must be >= 1", B);
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_INVALID, "E = %d outside [1, %d]", E, MOE_MAX_EXPERTS);
  if (num_gpus < 1 || num_gpus > moe::kEplbMaxGpus)
    return fail(MOE_ERR_INVALID, "num_gpus = %d outside [1, %d]", num_gpus, moe::kEplbMaxGpus);
  if (num_phys < E || num_phys > moe::kEplbMaxPhys || num_phys % num_gpus != 0)
    return fail(MOE_ERR_INVALID, "num_phys = %d must be in [E, %d] and a multiple of num_gpus", num_phys, moe::kEplbMaxPhys);
  if (num_nodes < 1 || num_gpus % num_nodes != 0)
    return fail(MOE_ERR_INVALID, "num_nodes = %d must divide num_gpus = %d", num_nodes, num_gpus);
  if (num_groups < 0 || (num_groups > 0 && E % num_groups != 0))
    return fail(MOE_ERR_INVALID, "num_groups = %d must be 0 or divide E = %d", num_groups, E);
  if (!aligned(loads, 4) || !aligned(phy2log, 4) || !aligned(log_count, 4) || !aligned(gpu_load, 4))
    return fail(MOE_ERR_INVALID, "an EPLB array is not 4-byte aligned");
  moe::EplbParams p;
  p.loads = loads;
  p.B = B;
  p.E = E;
  p.num_phys = num_phys;
  p.num_gpus = num_gpus;
  p.num_nodes = num_nodes;
  p.num_groups = num_groups;
  p.hier = num_groups > 0 && num_groups % num_nodes == 0;
  p.phy2log = phy2log;
  p.log_count = log_count;
  p.gpu_load = gpu_load;
  cudaError_t e = moe::launch_eplb_plan(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "eplb_plan launch");
  return MOE_OK;
}

moe_status taot_match_batched(const int32_t* expert_loads, const float* plan, int32_t B, int32_t E,
                              int32_t R, int32_t ranks_per_node, int32_t K,
                              int32_t* slot_expert, int32_t* slot_tokens, int32_t* rank_load,
                              moe_stream_t stream) {
  if (!expert_loads || !plan || !rank_load || (K > 0 && (!slot_expert || !slot_tokens)))
    return fail(MOE_ERR_INVALID, "a matching argument is NULL");
  if (B < 1) return fail(MOE_ERR_INVALID, "B = %d must be >= 1", B);
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_INVALID, "E = %d outside [1, %d]", E, MOE_MAX_EXPERTS);
  if (R < 1 || R > MOE_MAX_RANKS || E % R != 0) return fail(MOE_ERR_INVALID, "R = %d must be in [1, %d] and divide E", R, MOE_MAX_RANKS);
  if (ranks_per_node < 1 || R % ranks_per_node != 0) return fail(MOE_ERR_INVALID, "ranks_per_node = %d must divide R", ranks_per_node);
  if (K < 0 || K > moe::kMatchMaxRounds) return fail(MOE_ERR_INVALID, "K = %d outside [0, %d]", K, moe::kMatchMaxRounds);
  if (!aligned(expert_loads, 4) || !aligned(plan, 4) || !aligned(slot_expert, 4) || !aligned(slot_tokens, 4) || !aligned(rank_load, 4))
    return fail(MOE_ERR_INVALID, "a matching array is not 4-byte aligned");
  moe::MatchParams p;
  p.expert_loads = expert_loads;
  p.plan = plan;
  p.B = B;
  p.E = E;
  p.R = R;
  p.ranks_per_node = ranks_per_node;
  p.K = K;
  p.slot_expert = slot_expert;
  p.slot_tokens = slot_tokens;
  p.rank_load = rank_load;
  cudaError_t e = moe::launch_taot_match(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "taot_match launch");
  return MOE_OK;
}

moe_status moe_router_combine(const int32_t* counts, const float* P, const int64_t* T_shard, int32_t G,
                              int32_t E, int32_t k, float alpha, int32_t n_ranks, int32_t masked_p,
                              int32_t* counts_out, float* f, float* P_out, float* scalars, int32_t* rank_load,
                              moe_stream_t stream) {
  if (!counts || !P || !T_shard) return fail(MOE_ERR_INVALID, "a shard input is NULL");
  if (G < 1 || G > moe::kMaxShards) return fail(MOE_ERR_INVALID, "G = %d outside [1, %d]", G, moe::kMaxShards);
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_INVALID, "E = %d outside [1, %d]", E, MOE_MAX_EXPERTS);
  if (k < 1 || k > MOE_MAX_TOPK || k > E) return fail(MOE_ERR_INVALID, "k = %d outside [1, min(E, %d)]", k, MOE_MAX_TOPK);
  if (!(alpha >= 0.f) || !std::isfinite(alpha)) return fail(MOE_ERR_INVALID, "alpha must be finite and >= 0");
  if (n_ranks < 0 || n_ranks > MOE_MAX_RANKS || (n_ranks > 0 && E % n_ranks != 0))
    return fail(MOE_ERR_INVALID, "n_ranks = %d must be 0 or a divisor of E in [1, %d]", n_ranks, MOE_MAX_RANKS);
  if (!counts_out || !f || !P_out || !scalars || (n_ranks > 0 && !rank_load))
    return fail(MOE_ERR_INVALID, "a combined output is NULL");
  if (!aligned(counts, 4) || !aligned(P, 4) || !aligned(counts_out, 4) || !aligned(f, 4) || !aligned(P_out, 4) ||
      !aligned(scalars, 4) || (rank_load && !aligned(rank_load, 4)))
    return fail(MOE_ERR_INVALID, "an array is not 4-byte aligned");
  moe::CombineParams p;
  std::memset(&p, 0, sizeof(p));
  long long T = 0;
  for (int g = 0; g < G; ++g) {
    if (T_shard[g] < 0 || T_shard[g] >= (int64_t(1) << 31)) return fail(MOE_ERR_INVALID, "T_shard[%d] = %lld outside [0, 2^31)", g, (long long)T_shard[g]);
    T += T_shard[g];
    p.T_shard[g] = double(T_shard[g]);
  }
  if (T < 1 || T * (long long)k >= (1ll << 31)) return fail(MOE_ERR_INVALID, "the shards' total T = %lld must be >= 1 with T*k < 2^31", T);
  p.counts = counts;
  p.P = P;
  p.G = G;
  p.E = E;
  p.k = k;
  p.T = T;
  p.alpha = alpha;
  p.n_ranks = n_ranks;
  p.masked_p = masked_p != 0;
  p.counts_out = counts_out;
  p.f = f;
  p.P_out = P_out;
  p.scalars = scalars;
  p.rank_load = rank_load;
  cudaError_t e = moe::launch_router_combine(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "router_combine launch");
  return MOE_OK;
}

moe_status moe_router_fwd_ex(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                             float alpha, int32_t renorm, int32_t n_ranks,
                             const float* bias, int32_t masked_p, float bias_gamma, float* bias_out,
                             int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                             float* scalars, int32_t* rank_load,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_router_args(logits, dt, T, E, k);
  if (s != MOE_OK) return s;
  if ((s = check_fwd_outputs(k, alpha, renorm, n_ranks, E, idx, gate, counts, f, P, scalars, rank_load)) != MOE_OK) return s;
  if ((s = check_ws(ws, ws_bytes, E)) != MOE_OK) return s;
  if (!std::isfinite(bias_gamma)) return fail(MOE_ERR_INVALID, "bias_gamma must be finite");
  if ((bias && !aligned(bias, 4)) || (bias_out && !aligned(bias_out, 4))) return fail(MOE_ERR_INVALID, "bias is not 4-byte aligned");
  // the extended step's forward alone: the persistent kernel in mode kModeFwdExt
  const RouterVariant* v = pick_variant(dt, E, aligned(logits, 16));
  if (!v) return fail(MOE_ERR_INVALID, "no kernel variant for E = %d", E);
  const moe::StepExtVariant* xv = step_ext_variant(dt, v);
  if (!xv) return fail(MOE_ERR_INVALID, "no extended forward kernel for E = %d", E);
  RouterParams p = base_params(logits, T, E, k);
  p.alpha = alpha;
  p.renorm = renorm < 0 ? (k > 1) : renorm;
  p.n_ranks = n_ranks;
  p.bias = bias;
  p.bias_gamma = bias_gamma;
  p.bias_out = bias_out;
  p.masked_p = masked_p != 0;
  p.idx = idx; p.gate = gate; p.counts = counts; p.f = f; p.P = P; p.scalars = scalars; p.rank_load = rank_load;
  bind_ws(p, ws, E);
  Geometry geo;
  if ((s = persistent_geometry(v, dt, T, E, k, false, &geo, xv->fwd_ext)) != MOE_OK) return s;
  p.G = geo.G;
  p.n_groups = (p.G + moe::kGroupCtas - 1) / moe::kGroupCtas;
  p.rows_per_stage = geo.rows_per_stage;
  p.n_slots = geo.n_slots;
  p.asg_cap = geo.asg_cap;
  p.rstat_cap = geo.rstat_cap;
  return launch_persistent(xv->fwd_ext, p, geo.smem, stream);
}

moe_status moe_router_bwd_full(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                               float alpha, const float* f, float grad_scale, int32_t masked_p,
                               const int32_t* idx, const float* dgate, int32_t renorm,
                               float* dlogits, moe_stream_t stream) {
  moe_status s = check_router_args(logits, dt, T, E, k);
  if (s != MOE_OK) return s;
  if (!(alpha >= 0.f) || !std::isfinite(alpha)) return fail(MOE_ERR_INVALID, "alpha must be finite and >= 0");
  if (!std::isfinite(grad_scale)) return fail(MOE_ERR_INVALID, "grad_scale must be finite");
  if (renorm < -1 || renorm > 1) return fail(MOE_ERR_INVALID, "renorm must be -1, 0 or 1");
  if (!f || !dlogits) return fail(MOE_ERR_INVALID, "f or dlogits is NULL");
  if ((dgate || masked_p) && !idx) return fail(MOE_ERR_INVALID, "idx is NULL but dgate or masked_p needs the picks");
  if (!aligned(dlogits, 4) || !aligned(f, 4) || (idx && !aligned(idx, 4)) || (dgate && !aligned(dgate, 4)))
    return fail(MOE_ERR_INVALID, "an array is not 4-byte aligned");
  const moe::ExtVariant* v = pick_ext_variant(dt, E, aligned(logits, 16) && aligned(dlogits, 16));
  if (!v) return fail(MOE_ERR_INVALID, "no kernel variant for E = %d", E);
  DeviceInfo d;
  int dev = 0;
  if ((s = device_info(&d, &dev)) != MOE_OK) return s;
  int blocks = 0;
  if ((s = occupancy(v->bwd, moe::kExtBwdThreads, 0, dev, &blocks)) != MOE_OK) return s;
  const int64_t rows_per_block = int64_t(moe::kExtBwdThreads / moe::kWarp) * (moe::kWarp / v->LPR);
  const int64_t want = (T + rows_per_block - 1) / rows_per_block;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(blocks) * d.sms)));
  moe::BwdFullParams p;
  std::memset(&p, 0, sizeof(p));
  p.logits = logits;
  p.T = T;
  p.E = E;
  p.k = k;
  p.f = f;
  p.masked_p = masked_p != 0;
  p.coef = float(double(grad_scale) * double(alpha) * double(E) / (masked_p ? double(T) * double(k) : double(T)));
  p.idx = idx;
  p.dgate = dgate;
  p.renorm = renorm < 0 ? (k > 1) : renorm;
  p.dlogits = dlogits;
  void* args[] = {&p};
  cudaError_t e = cudaLaunchKernel(v->bwd, dim3(grid), dim3(moe::kExtBwdThreads), args, 0, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernel");
  return MOE_OK;
}

void moe_set_trace_buffer(uint64_t* device_buf, int32_t max_ctas) {
  g_trace_ctas.store(device_buf ? max_ctas : 0, std::memory_order_relaxed);
  g_trace.store(reinterpret_cast<unsigned long long*>(device_buf), std::memory_order_relaxed);
}

void moe_set_unreachable_barriers(int32_t enable) { g_barrier_extra.store(enable ? 1u : 0u, std::memory_order_relaxed); }

void moe_set_wait_timeout_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs, std::memory_order_relaxed); }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

int32_t moe_abi_version(void) { return MOE_ROUTER_ABI_VERSION; }

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_router_step_static: moe_router_step without a caller workspace.
//
// Some callers cannot hand the library any device memory of their own: code
// that runs where allocating is not allowed or not safe (for instance while a
// host thread must not block on the allocator, inside plugins whose memory
// budget is fixed when they are loaded, or from runtimes that own every byte
// of device memory through their own pool and expose no allocator to native
// code).  For them this entry point keeps its scratch in a fixed array that is
// part of the library image: every GPU that loads the library holds it, all
// kStaticScratchBytes of it, until the process exits, and the call itself
// allocates nothing.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = (size_t(4) << 20) + (size_t(768) << 10);   // 4.75 MiB
constexpr int kStaticMaxExperts = 512;      // ws_layout(512).total fits in kStaticScratchBytes
static_assert(kStaticScratchBytes >= 4096 + kGroupHistBytes + kPfixBytes + size_t(kStaticMaxExperts) * 4 * (2 * 1024 + 1),
              "scratch size");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up once
// per device (with that device current) and cached.
moe_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_INVALID, "device %d is beyond the %d this entry point serves", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_router_step_static(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                                             float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                                             float grad_scale,
                                             int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                                             float* scalars, int32_t* rank_load,
                                             int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                             int32_t* n_dropped, float* dlogits, moe_stream_t stream) {
  if (E > kStaticMaxExperts)
    return fail(MOE_ERR_INVALID, "moe_router_step_static serves at most %d experts (E = %d); use moe_router_step",
                kStaticMaxExperts, E);
  // Every argument is checked before anything is queued on the stream, so a
  // refused call leaves the shared array as it was.
  moe_status s = check_step_args(logits, dt, T, E, k, alpha, renorm, n_ranks, capacity_factor, grad_scale, idx, gate,
                                 counts, f, P, scalars, rank_load, perm, slot, offsets, kept, n_dropped, dlogits);
  if (s != MOE_OK) return s;
  void* ws = nullptr;
  if ((s = static_scratch(&ws)) != MOE_OK) return s;
  const size_t need = ws_layout(E).total;
  if (need > kStaticScratchBytes) return fail(MOE_ERR_INVALID, "E = %d needs %zu bytes of scratch", E, need);
  // The array keeps the previous call's contents.  The barrier's arrival
  // count (the low half of the control block's first word), the other
  // counters and the group sums must start at zero; the rest is written
  // before it is read.  The error bits (the first word's high half) are left
  // as they are: after an expired wait they stay set, later calls write
  // nothing, and moe_get_device_status(NULL, ...) reads and clears them.
  static_assert(offsetof(moe::Ctrl, sync) == 0 && offsetof(moe::Ctrl, done) == 8, "control block layout");
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(static_cast<unsigned char*>(ws) + offsetof(moe::Ctrl, done), 0,
                        ws_layout(E).tile_hist - offsetof(moe::Ctrl, done), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return moe_router_step(logits, dt, T, E, k, alpha, renorm, n_ranks, capacity_factor, grad_scale, idx, gate, counts,
                         f, P, scalars, rank_load, perm, slot, offsets, kept, n_dropped, dlogits, ws, need, stream);
}
