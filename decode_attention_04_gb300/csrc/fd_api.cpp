// Host side of libfd.so: argument checks, the split plan, the library-owned
// workspace, and the exported C entry points declared in fd_decode_attn.h.

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "fd_decode_attn.h"
#include "fd_internal.h"

namespace {

constexpr int kMaxGroup = 16;

// Test hook (fd_debug_withhold_copies): the tile index from which split blocks
// issue no copies; INT_MAX: off.
std::atomic<int> g_withhold_tile{INT_MAX};

bool supported_hs(int HS) { return HS == 64 || HS == 128 || HS == 256 || HS == 512; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int B, int NH, int NKV, int HS, int capacity, int window) {
  if (B < 0 || NH <= 0 || NKV <= 0 || capacity <= 0) return FD_ERR_INVALID_ARG;
  if (window > capacity) return FD_ERR_INVALID_ARG;
  if (B > 65535 || NKV > 65535) return FD_ERR_INVALID_ARG;  // grid y/z limits
  if (!supported_hs(HS)) return FD_ERR_UNSUPPORTED;
  if (NH % NKV != 0 || NH / NKV > kMaxGroup) return FD_ERR_UNSUPPORTED;
  return FD_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Partial slots per row: one per block, or one per cluster of blocks.
int slots(const fd_plan_t& p) { return p.num_splits / (p.cluster > 0 ? p.cluster : 1); }

// Workspace layout:
//   [counters: B*NKV uint32 split counters when a row has more than one
//    partial slot (followed by B*NKV count-out words for the group step), then
//    one work-item counter for a persistent grid; zero before the first call]
//   [O partials: fp32 B*NH*slots*HS] [(m, l): fp32 B*NH*slots*2]   (slots > 1)
// each part rounded up to 256 bytes.
long long split_counter_words(const fd_plan_t& p) {
  return slots(p) > 1 ? static_cast<long long>(p.B) * p.NKV * (p.fused == 2 ? 2 : 1) : 0;
}

size_t ws_counter_bytes(const fd_plan_t& p) {
  const long long words = split_counter_words(p) + (p.persistent > 0 ? 1 : 0);
  return words ? round_up(static_cast<size_t>(words) * sizeof(unsigned int), 256) : 0;
}

size_t ws_o_bytes(const fd_plan_t& p) {
  return round_up(static_cast<size_t>(p.B) * p.NH * slots(p) * p.HS * sizeof(float), 256);
}

size_t ws_total(const fd_plan_t& p) {
  if (slots(p) <= 1) return ws_counter_bytes(p);
  return ws_counter_bytes(p) + ws_o_bytes(p) +
         round_up(static_cast<size_t>(p.B) * p.NH * slots(p) * 2 * sizeof(float), 256);
}

// Work items of the split grid: one per (split, KV head, sequence).
long long work_items(const fd_plan_t& p) { return static_cast<long long>(p.num_splits) * p.NKV * p.B; }

// A persistent split grid (a fixed set of blocks taking work items from a
// device counter) is available for the tensor-core kernel without clusters
// or the fused merge.
bool persistent_allowed(const fd_plan_t& p) {
  const long long items = work_items(p);
  return p.path == FD_PATH_TC && p.cluster == 1 && !p.fused && items >= 1 && items <= (1ll << 30);
}

// Blocks of a persistent grid: every resident block slot once, or one per
// item when there are fewer items.
int persistent_blocks(const fd_plan_t& p) {
  const long long slots_gpu = static_cast<long long>(p.num_sms) * p.ctas_per_sm;
  return static_cast<int>(std::max(1ll, std::min(work_items(p), slots_gpu)));
}

// Off by default: measured on GB300 (us per layer, graph of layers, one
// block per split -> persistent), the two multi-wave workloads barely moved
// (ragged d128 batch 168.0 -> 167.8, or 166.7 at twice the splits; MQA long
// 174.8 -> 172.5; E4M3 MQA long 122.9 -> 126.5) and one-wave grids lost
// (ring 7.42 -> 9.17, llama tiny 5.84 -> 6.92): the hardware already starts a
// new block as soon as one retires, and the persistent kernel holds more
// registers, which keeps the merge kernel's early blocks off the SMs.
int persistent_rule(const fd_plan_t& p) {
  (void)p;
  return 0;
}

// Fused merge, mode 1 (the last split block of each (sequence, KV head)
// merges) when the group's partials, which that one block reads, stay within
// 256 KB; mode 2 (every block of a group waits for the group, then merges a
// share) when the whole grid is resident at once on the plan's SMs.
bool fused_rule_allowed(const fd_plan_t& p, int mode = 1) {
  const long long G = p.NH / p.NKV;
  if (p.path != FD_PATH_TC || p.cluster != 1 || slots(p) <= 1) return false;
  if (mode == 2)
    return static_cast<long long>(p.B) * p.NKV * p.num_splits <= static_cast<long long>(p.num_sms) * p.ctas_per_sm;
  return G * p.num_splits * p.HS * static_cast<long long>(sizeof(float)) <= (256ll << 10);
}

// Off by default: measured on GB300 (us per layer), the separate merge kernel,
// whose blocks programmatic dependent launch makes resident early, beat both
// in-launch forms on the ring (6.14 against 7.27 for the last block, 7.07 for
// the group step), MQA 4k (8.81 against 11.85 for the group step) and MQA 32k
// (19.25 against 22.12); only Llama tiny favoured the last block (4.79 against
// 4.88). Split blocks that wait for their group, or for the last block, hold
// their SM slots, so the next layer's blocks cannot start early. Kept as
// options (fd_plan_override) and tested.
int fused_rule(const fd_plan_t& p) {
  (void)p;
  return 0;
}

// 4 KB copy groups (a tile that needs the whole SM) only for the head-dim-512,
// 16-row tile, and only when the grid fits one wave at one block per SM.
// E4M3 groups: 2 KB (1 KB for head dim 256, whose small sliding bands want
// short tiles).
int group_rule(const fd_plan_t& p) {
  const long long G = p.NH / p.NKV;
  const long long blocks = static_cast<long long>(p.B) * p.NKV * p.num_splits;
  if (p.path == FD_PATH_UMMA) return 16384;  // one TMA box: 128 positions x 64 dims
  if (p.kv_dtype == FD_KV_E4M3) {
    // 1 KB groups for head dim 256 with more than 8 query rows, and for 64 /
    // 128 when the plan cut the band into whole short tiles
    const int short_tile = fd::tc_short_tile_positions(p.HS);
    return ((p.HS == 256 && G > 8) || (short_tile > 0 && p.granule == short_tile)) ? 1024 : 2048;
  }
  if (p.path == FD_PATH_TC && p.HS == 256 && G <= 8) return 4096;  // the sliding ring's tile
  return (p.path == FD_PATH_TC && p.HS == 512 && G > 8 && blocks <= p.num_sms) ? 4096 : 2048;
}

// Consumer warps of the tensor-core tile: fixed per (cache type, head dim,
// G <= 8 or not), except the E4M3 head-dim-512, 16-row tile: eight warps when
// the grid is one block per SM, four when blocks share SMs. 0 on the SIMT path.
bool warps_choice_open(const fd_plan_t& p) {
  return p.path == FD_PATH_TC && p.kv_dtype == FD_KV_E4M3 && p.HS == 512 && p.NH / p.NKV > 8;
}

int warps_rule(const fd_plan_t& p) {
  if (p.path == FD_PATH_UMMA) return 4;  // softmax warps; one more issues the MMAs
  if (p.path != FD_PATH_TC) return 0;
  const bool two = p.NH / p.NKV > 8;
  if (p.kv_dtype == FD_KV_E4M3) {
    if (p.HS == 64) return 2;
    if (p.HS == 128) return 4;
    if (p.HS == 256) return 8;
    const long long blocks = static_cast<long long>(p.B) * p.NKV * p.num_splits;
    return two && blocks <= p.num_sms ? 8 : 4;
  }
  return (p.HS == 256 || (p.HS == 512 && two)) ? 8 : 4;
}

void finish_plan(fd_plan_t* p, int fused = -1, int persistent = -1) {
  p->fused = fused < 0 ? fused_rule(*p) : (fused > 0 && fused_rule_allowed(*p, fused) ? fused : 0);
  p->persistent = persistent < 0 ? persistent_rule(*p)
                                 : (persistent && persistent_allowed(*p) ? persistent_blocks(*p) : 0);
  p->group_bytes = group_rule(*p);
  p->consumer_warps = warps_rule(*p);
  p->workspace_bytes = ws_total(*p);
  p->workspace_zero_bytes = ws_counter_bytes(*p);
}

bool valid_kv(int kv_dtype, int path) {
  return kv_dtype == FD_KV_BF16 || (kv_dtype == FD_KV_E4M3 && path == FD_PATH_TC);
}

bool valid_path(const fd_plan_t& p) {
  if (p.path == FD_PATH_TC || p.path == FD_PATH_SIMT) return true;
  return p.path == FD_PATH_UMMA && p.kv_dtype == FD_KV_BF16 && fd::umma_shape_ok(p.HS, p.NH / p.NKV, p.window);
}

bool valid_cluster(int cluster, int num_splits, int HS, int path) {
  if (cluster < 1 || cluster > 16 || (cluster & (cluster - 1)) != 0) return false;
  if (num_splits % cluster != 0 || (HS / cluster) % 4 != 0) return false;
  return cluster == 1 || path == FD_PATH_TC;
}

// The split rule, documented in fd_decode_attn.h beside fd_plan_t.
int make_plan(int B, int NH, int NKV, int HS, int capacity, int window, int max_len, int num_sms,
              int ctas_per_sm, int max_cluster, int path, int kv_dtype, fd_plan_t* plan) {
  if (!plan) return FD_ERR_INVALID_ARG;
  int rc = check_shape(B, NH, NKV, HS, capacity, window);
  if (rc != FD_OK) return rc;
  if (num_sms <= 0 || ctas_per_sm <= 0 || max_cluster < 1) return FD_ERR_INVALID_ARG;
  if (path == FD_PATH_AUTO) path = FD_PATH_TC;
  if (path != FD_PATH_TC && path != FD_PATH_SIMT) return FD_ERR_INVALID_ARG;
  if (kv_dtype != FD_KV_BF16 && kv_dtype != FD_KV_E4M3) return FD_ERR_INVALID_ARG;
  if (!valid_kv(kv_dtype, path)) return FD_ERR_UNSUPPORTED;

  const int keep = window > 0 ? window : capacity;
  int max_band = keep < capacity ? keep : capacity;
  if (max_len > 0 && max_len < max_band) max_band = max_len;
  if (max_band < 1) max_band = 1;

  const long long units = static_cast<long long>(B > 0 ? B : 1) * NKV;
  // With large query groups a partial (G x HS floats) is costly next to a
  // split's K/V bytes, so fill each SM once rather than with every resident
  // block.
  const int G = NH / NKV;
  const long long slots = static_cast<long long>(num_sms) * (G >= 8 ? 1 : ctas_per_sm);
  long long s_fill = (slots + units - 1) / units;
  if (s_fill < 1) s_fill = 1;
  // Whole-tile splits where filling the GPU would cut the band into pieces of
  // under two tiles; longer pieces keep single positions as the granule, so
  // rounding never leaves SMs idle.
  const int tile = fd::plan_granule(path, HS, kv_dtype == FD_KV_E4M3);
  int granule = (max_band + s_fill - 1) / s_fill < 2 * tile ? tile : 1;
  // An E4M3 cache with head dim 64 or 128 has a half-length tile (1 KB copy
  // groups) for such short bands: twice the blocks for the same band.
  const int short_tile = fd::tc_short_tile_positions(HS);
  if (kv_dtype == FD_KV_E4M3 && path == FD_PATH_TC && granule == tile && short_tile > 0) granule = short_tile;
  auto chunk_for = [&](long long S) {
    long long c = (max_band + S - 1) / S;
    c = (c + granule - 1) / granule * granule;
    return c < granule ? static_cast<long long>(granule) : c;
  };
  long long chunk = chunk_for(s_fill);
  // Balance bound: at most ~2 MiB of K+V per split, so a ragged batch does not
  // leave a few long splits running alone at the end.
  const long long pos_bytes = (kv_dtype == FD_KV_E4M3 ? 2ll : 4ll) * HS;  // K + V bytes per position
  long long bound_bytes = 2ll << 20;
  // With large query groups, a band too long for one block per SM first fills
  // every resident block slot once, with twice the bound, before adding waves
  // (measured: bf16 MQA, 4 x 131072 positions, 76 splits in one wave 164.9 us
  // per layer against 152 splits in two 170.0).
  if (G >= 8 && chunk * pos_bytes > bound_bytes && ctas_per_sm > 1) {
    s_fill = std::max<long long>(1, (static_cast<long long>(num_sms) * ctas_per_sm + units - 1) / units);
    granule = (max_band + s_fill - 1) / s_fill < 2 * tile ? tile : 1;
    chunk = chunk_for(s_fill);
    bound_bytes = 4ll << 20;
  }
  const long long max_chunk = std::max<long long>(granule, bound_bytes / pos_bytes);
  long long S = (max_band + chunk - 1) / chunk;
  if (chunk > max_chunk) {
    long long waves = (static_cast<long long>(max_band) + max_chunk * s_fill - 1) / (max_chunk * s_fill);
    S = waves * s_fill;
    chunk = chunk_for(S);
    S = (max_band + chunk - 1) / chunk;
  }
  if (S < 1) S = 1;
  if (S > 65535 * 64) S = 65535 * 64;

  // No clusters by default: a cluster must find `cluster` free block slots in
  // one GPC at once, and on GB300 that stranded slots and cost more than the
  // smaller partials saved (measured on every workload here). Clusters remain
  // available through fd_plan_override.
  const int cluster = 1;

  fd_plan_t p{};
  p.num_splits = static_cast<int>(S);
  p.path = path;
  p.cluster = cluster;
  p.max_cluster = max_cluster;
  p.granule = granule;
  p.max_band = max_band;
  p.ctas_per_sm = ctas_per_sm;
  p.num_sms = num_sms;
  p.B = B;
  p.NH = NH;
  p.NKV = NKV;
  p.HS = HS;
  p.capacity = capacity;
  p.window = window;
  p.kv_dtype = kv_dtype;
  finish_plan(&p);
  *plan = p;
  return FD_OK;
}

// Per-device SM count, cached.
std::mutex g_mu;
std::map<int, int> g_sms;

int device_sms(int device, int* sms) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sms.find(device);
    if (it != g_sms.end()) {
      *sms = it->second;
      return FD_OK;
    }
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0)
    return FD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  g_sms[device] = v;
  *sms = v;
  return FD_OK;
}

// Resident split blocks per SM and the largest schedulable cluster of the
// tensor-core kernel for (device, HS, G, cache type): occupancy queries,
// made once and cached (they sit on every fd_decode_attn call's host path).
struct Occupancy {
  int ctas = 0;
  int max_cluster = 1;
};
std::map<std::tuple<int, int, int, bool>, Occupancy> g_occ;

int device_occupancy(int device, int HS, int G, bool kv8, int* ctas, int* max_cluster) {
  const auto key = std::make_tuple(device, HS, G, kv8);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) {
      *ctas = it->second.ctas;
      *max_cluster = it->second.max_cluster;
      return FD_OK;
    }
  }
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return FD_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return FD_ERR_CUDA;
  Occupancy o;
  cudaError_t e = fd::query_ctas_per_sm(FD_PATH_TC, HS, G, kv8, &o.ctas);
  if (e == cudaSuccess) e = fd::query_max_cluster(HS, G, kv8, &o.max_cluster);
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess || o.ctas <= 0) return FD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  g_occ[key] = o;
  *ctas = o.ctas;
  *max_cluster = o.max_cluster;
  return FD_OK;
}

// Library-owned workspaces, one per (device, stream), grow-only.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

int get_workspace(int device, cudaStream_t stream, size_t need, void** ptr) {
  *ptr = nullptr;
  if (need == 0) return FD_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_ws[{device, reinterpret_cast<uintptr_t>(stream)}];
  if (w.bytes >= need) {
    *ptr = w.ptr;
    return FD_OK;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return FD_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return FD_ERR_WORKSPACE;
  // The stream may still use the old buffer: finish its work before freeing.
  if (w.ptr) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FD_ERR_CUDA;
    cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, need) != cudaSuccess) return FD_ERR_CUDA;
  // The counters must start at zero: clear on the call's stream, ahead of the
  // call's kernels (a plain cudaMemset would run on the legacy stream, which a
  // non-blocking stream is not ordered with).
  if (cudaMemsetAsync(p, 0, need, stream) != cudaSuccess) {
    cudaFree(p);
    return FD_ERR_CUDA;
  }
  w.ptr = p;
  w.bytes = need;
  *ptr = p;
  return FD_OK;
}

// k_scale / v_scale are null for a bf16 cache; for an E4M3 cache k_cache and
// v_cache hold the codes.
int run(const fd_plan_t& plan, void* workspace, size_t workspace_bytes, float* out_f32, const void* q,
        const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale, void* out,
        const int* lens, float scale, cudaStream_t stream) {
  if (plan.B == 0) return FD_OK;
  const bool kv8 = plan.kv_dtype == FD_KV_E4M3;
  if (!q || !k_cache || !v_cache || !out || !lens) return FD_ERR_INVALID_ARG;
  if (kv8 && (!k_scale || !v_scale)) return FD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lens, 4) || (out_f32 && !aligned(out_f32, 16)) ||
      (kv8 && (!aligned(k_scale, 4) || !aligned(v_scale, 4))))
    return FD_ERR_ALIGNMENT;
  const size_t need = ws_total(plan);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return FD_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return FD_ERR_ALIGNMENT;
  }
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(plan.HS));

  fd::LaunchArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.kv8 = kv8 ? 1 : 0;
  if (kv8) {
    a.k8 = static_cast<const uint8_t*>(k_cache);
    a.v8 = static_cast<const uint8_t*>(v_cache);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
  } else {
    a.k = static_cast<const uint16_t*>(k_cache);
    a.v = static_cast<const uint16_t*>(v_cache);
  }
  a.out = static_cast<uint16_t*>(out);
  a.out_f32 = out_f32;
  a.lens = lens;
  char* ws = static_cast<char*>(workspace);
  a.counters = need ? reinterpret_cast<unsigned int*>(ws) : nullptr;
  a.persistent = plan.persistent;
  a.work_counter = plan.persistent > 0 ? a.counters + split_counter_words(plan) : nullptr;
  a.ws_o = need ? reinterpret_cast<float*>(ws + ws_counter_bytes(plan)) : nullptr;
  a.ws_ml = need ? reinterpret_cast<float*>(ws + ws_counter_bytes(plan) + ws_o_bytes(plan)) : nullptr;
  a.fused = plan.fused;
  a.group_bytes = plan.group_bytes;
  a.consumer_warps = plan.consumer_warps;
  a.B = plan.B;
  a.NH = plan.NH;
  a.NKV = plan.NKV;
  a.HS = plan.HS;
  a.capacity = plan.capacity;
  a.window = plan.window;
  a.num_splits = plan.num_splits;
  a.cluster = plan.cluster;
  a.granule = plan.granule;
  a.path = plan.path;
  a.min_len = plan.min_len;
  a.withhold_tile = g_withhold_tile.load(std::memory_order_relaxed);
  // whole-tile splits that cover the plan's band bound: one tile per block (a
  // longer band than the bound stays exact, its blocks just take two tiles)
  a.one_tile = plan.path == FD_PATH_TC && plan.persistent == 0 && plan.granule > 1 &&
               static_cast<long long>(plan.max_band) <= static_cast<long long>(plan.num_splits) * plan.granule;
  a.scale_log2 = scale * 1.4426950408889634f;
  return fd::launch_decode(a, stream) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // namespace

extern "C" {

int fd_plan_sms(int B, int NH, int NKV, int HS, int capacity, int window, int max_len, int num_sms,
                int ctas_per_sm, int max_cluster, fd_plan_t* plan) {
  return make_plan(B, NH, NKV, HS, capacity, window, max_len, num_sms, ctas_per_sm, max_cluster, FD_PATH_AUTO,
                   FD_KV_BF16, plan);
}

int fd_plan_sms_kv(int B, int NH, int NKV, int HS, int capacity, int window, int max_len, int num_sms,
                   int ctas_per_sm, int max_cluster, int kv_dtype, fd_plan_t* plan) {
  return make_plan(B, NH, NKV, HS, capacity, window, max_len, num_sms, ctas_per_sm, max_cluster, FD_PATH_AUTO,
                   kv_dtype, plan);
}

int fd_plan_kv(int B, int NH, int NKV, int HS, int capacity, int window, int max_len, int device, int kv_dtype,
               fd_plan_t* plan) {
  if (kv_dtype != FD_KV_BF16 && kv_dtype != FD_KV_E4M3) return FD_ERR_INVALID_ARG;
  if (!plan) return FD_ERR_INVALID_ARG;
  int rc = check_shape(B, NH, NKV, HS, capacity, window);
  if (rc != FD_OK) return rc;
  int sms = 0;
  rc = device_sms(device, &sms);
  if (rc != FD_OK) return rc;
  int ctas = 0, max_cluster = 1;
  rc = device_occupancy(device, HS, NH / NKV, kv_dtype == FD_KV_E4M3, &ctas, &max_cluster);
  if (rc != FD_OK) return rc;
  return make_plan(B, NH, NKV, HS, capacity, window, max_len, sms, ctas, max_cluster, FD_PATH_AUTO, kv_dtype,
                   plan);
}

int fd_plan(int B, int NH, int NKV, int HS, int capacity, int window, int max_len, int device,
            fd_plan_t* plan) {
  return fd_plan_kv(B, NH, NKV, HS, capacity, window, max_len, device, FD_KV_BF16, plan);
}

int fd_plan_override(fd_plan_t* plan, int num_splits, int path, int cluster, int fused) {
  if (!plan || num_splits < 0 || cluster < 0 || num_splits > 65535 * 64) return FD_ERR_INVALID_ARG;
  if (path != FD_PATH_AUTO && path != FD_PATH_SIMT && path != FD_PATH_TC && path != FD_PATH_UMMA)
    return FD_ERR_INVALID_ARG;
  if (check_shape(plan->B, plan->NH, plan->NKV, plan->HS, plan->capacity, plan->window) != FD_OK)
    return FD_ERR_INVALID_ARG;
  fd_plan_t p = *plan;
  if (path != FD_PATH_AUTO && path != p.path) {
    p.path = path;
    // a forced kernel family walks single-position chunks; the tensor-memory
    // kernel 16-position ones (one P.V step), so only the band's last split
    // has rows that do not fill its boxes or its last P.V step
    p.granule = path == FD_PATH_UMMA ? 16 : 1;
  }
  if (!valid_kv(p.kv_dtype, p.path) || !valid_path(p)) return FD_ERR_INVALID_ARG;
  if (num_splits > 0) p.num_splits = num_splits;
  if (cluster > 0) p.cluster = cluster;
  if (p.path == FD_PATH_SIMT && cluster == 0) p.cluster = 1;  // the SIMT path has no clusters
  if (!valid_cluster(p.cluster, p.num_splits, p.HS, p.path)) return FD_ERR_INVALID_ARG;
  if (fused > 2 || (fused > 0 && !fused_rule_allowed(p, fused))) return FD_ERR_INVALID_ARG;
  finish_plan(&p, fused);
  *plan = p;
  return FD_OK;
}

int fd_plan_persistent(fd_plan_t* plan, int persistent) {
  if (!plan || persistent < -1 || persistent > 1) return FD_ERR_INVALID_ARG;
  if (check_shape(plan->B, plan->NH, plan->NKV, plan->HS, plan->capacity, plan->window) != FD_OK)
    return FD_ERR_INVALID_ARG;
  fd_plan_t p = *plan;
  if (p.num_splits < 1 || !valid_path(p) || !valid_kv(p.kv_dtype, p.path) ||
      !valid_cluster(p.cluster, p.num_splits, p.HS, p.path) || p.num_sms < 1 || p.ctas_per_sm < 1)
    return FD_ERR_INVALID_ARG;
  if (persistent == 1 && !persistent_allowed(p)) return FD_ERR_INVALID_ARG;
  finish_plan(&p, p.fused, persistent);
  p.consumer_warps = plan->consumer_warps;  // a forced warp count stays
  p.group_bytes = plan->group_bytes;
  *plan = p;
  return FD_OK;
}

int fd_plan_min_len(fd_plan_t* plan, int min_len) {
  if (!plan || min_len < 0) return FD_ERR_INVALID_ARG;
  plan->min_len = min_len;
  return FD_OK;
}

size_t fd_workspace_bytes(const fd_plan_t* plan) { return plan ? ws_total(*plan) : 0; }

}  // extern "C"

namespace {

// A plan is usable for this call: it was made for these sizes and this cache
// type, and its fields are self-consistent.
int check_plan(const fd_plan_t* plan, int kv_dtype, int B, int NH, int NKV, int HS, int capacity, int window) {
  if (!plan) return FD_ERR_INVALID_ARG;
  int rc = check_shape(B, NH, NKV, HS, capacity, window);
  if (rc != FD_OK) return rc;
  if (plan->B != B || plan->NH != NH || plan->NKV != NKV || plan->HS != HS || plan->capacity != capacity ||
      plan->window != window || plan->kv_dtype != kv_dtype)
    return FD_ERR_INVALID_ARG;
  if (plan->num_splits < 1 || !valid_path(*plan) || plan->granule < 1 || !valid_kv(plan->kv_dtype, plan->path) || !valid_cluster(plan->cluster, plan->num_splits, plan->HS, plan->path) ||
      plan->fused < 0 || plan->fused > 2 || (plan->fused && !fused_rule_allowed(*plan, plan->fused)))
    return FD_ERR_INVALID_ARG;
  if (plan->min_len < 0) return FD_ERR_INVALID_ARG;
  if (plan->persistent < 0 ||
      (plan->persistent > 0 && (!persistent_allowed(*plan) || plan->persistent > work_items(*plan))))
    return FD_ERR_INVALID_ARG;
  if (plan->consumer_warps != warps_rule(*plan) &&
      !(warps_choice_open(*plan) && (plan->consumer_warps == 4 || plan->consumer_warps == 8)))
    return FD_ERR_INVALID_ARG;
  if (kv_dtype == FD_KV_E4M3 || plan->path == FD_PATH_UMMA)
    return plan->group_bytes == group_rule(*plan) ? FD_OK : FD_ERR_INVALID_ARG;
  if ((plan->group_bytes != 2048 && plan->group_bytes != 4096) ||
      (plan->group_bytes == 4096 && group_rule(*plan) != 4096 &&
       !(plan->HS == 512 && plan->NH / plan->NKV > 8 && plan->path == FD_PATH_TC)))
    return FD_ERR_INVALID_ARG;
  return FD_OK;
}

// Plan for the current device, take the library's workspace for this
// (device, stream), then run.
int run_auto(int kv_dtype, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
             const float* v_scale, void* out, const int* lens, int B, int NH, int NKV, int HS, int capacity,
             int window, float scale, fd_stream_t stream) {
  int rc = check_shape(B, NH, NKV, HS, capacity, window);
  if (rc != FD_OK) return rc;
  if (B == 0) return FD_OK;
  if (!q || !k_cache || !v_cache || !out || !lens) return FD_ERR_INVALID_ARG;
  if (kv_dtype == FD_KV_E4M3 && (!k_scale || !v_scale)) return FD_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FD_ERR_CUDA;
  fd_plan_t plan;
  rc = fd_plan_kv(B, NH, NKV, HS, capacity, window, 0, device, kv_dtype, &plan);
  if (rc != FD_OK) return rc;
  void* ws = nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = get_workspace(device, s, plan.workspace_bytes, &ws);
  if (rc != FD_OK) return rc;
  return run(plan, ws, plan.workspace_bytes, nullptr, q, k_cache, v_cache, k_scale, v_scale, out, lens, scale, s);
}

}  // namespace

extern "C" {

int fd_decode_attn_ex(const fd_plan_t* plan, void* workspace, size_t workspace_bytes, float* out_f32,
                      const void* q, const void* k_cache, const void* v_cache, void* out, const int* lens,
                      int B, int NH, int NKV, int HS, int capacity, int window, float scale,
                      fd_stream_t stream) {
  const int rc = check_plan(plan, FD_KV_BF16, B, NH, NKV, HS, capacity, window);
  if (rc != FD_OK) return rc;
  return run(*plan, workspace, workspace_bytes, out_f32, q, k_cache, v_cache, nullptr, nullptr, out, lens, scale,
             reinterpret_cast<cudaStream_t>(stream));
}

int fd_decode_attn(const void* q, const void* k_cache, const void* v_cache, void* out, const int* lens, int B,
                   int NH, int NKV, int HS, int capacity, int window, float scale, fd_stream_t stream) {
  return run_auto(FD_KV_BF16, q, k_cache, v_cache, nullptr, nullptr, out, lens, B, NH, NKV, HS, capacity, window,
                  scale, stream);
}

int fd_decode_attn_fp8_ex(const fd_plan_t* plan, void* workspace, size_t workspace_bytes, float* out_f32,
                          const void* q, const void* k8, const void* v8, const float* k_scale,
                          const float* v_scale, void* out, const int* lens, int B, int NH, int NKV, int HS,
                          int capacity, int window, float scale, fd_stream_t stream) {
  const int rc = check_plan(plan, FD_KV_E4M3, B, NH, NKV, HS, capacity, window);
  if (rc != FD_OK) return rc;
  return run(*plan, workspace, workspace_bytes, out_f32, q, k8, v8, k_scale, v_scale, out, lens, scale,
             reinterpret_cast<cudaStream_t>(stream));
}

int fd_decode_attn_fp8(const void* q, const void* k8, const void* v8, const float* k_scale, const float* v_scale,
                       void* out, const int* lens, int B, int NH, int NKV, int HS, int capacity, int window,
                       float scale, fd_stream_t stream) {
  return run_auto(FD_KV_E4M3, q, k8, v8, k_scale, v_scale, out, lens, B, NH, NKV, HS, capacity, window, scale,
                  stream);
}

int fd_debug_withhold_copies(int withhold_tile, unsigned long long wait_limit_ns) {
  const bool on = withhold_tile >= 0;
  const unsigned long long ns = on ? wait_limit_ns : 0;
  if (fd::set_wait_limit(ns) != cudaSuccess || fd::set_wait_limit_umma(ns) != cudaSuccess) return FD_ERR_CUDA;
  g_withhold_tile.store(on ? withhold_tile : INT_MAX, std::memory_order_relaxed);
  return FD_OK;
}

int fd_get_device_error(fd_stream_t stream, unsigned int* err) {
  if (!err) return FD_ERR_INVALID_ARG;
  return fd::read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream), err) == cudaSuccess
             ? FD_OK
             : FD_ERR_CUDA;
}

void fd_release(void) {
  fd::noalloc_forget();
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& kv : g_ws) {
    if (kv.second.ptr) {
      int prev = 0;
      cudaGetDevice(&prev);
      cudaSetDevice(kv.first.first);
      cudaFree(kv.second.ptr);
      cudaSetDevice(prev);
    }
  }
  g_ws.clear();
}

const char* fd_strerror(int status) {
  switch (status) {
    case FD_OK: return "ok";
    case FD_ERR_INVALID_ARG: return "invalid argument";
    case FD_ERR_UNSUPPORTED: return "unsupported shape (HS must be 64/128/256/512, NH % NKV == 0, NH/NKV <= 16)";
    case FD_ERR_ALIGNMENT: return "pointer not aligned (16 bytes for tensors and workspace, 4 for lens)";
    case FD_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case FD_ERR_WORKSPACE: return "workspace too small, or would need allocating while the stream is captured";
    case FD_ERR_SCRATCH_LIMIT:
      return "shape needs more split-partial scratch than the fixed 32 MiB array of fd_decode_attn_noalloc";
    default: return "unknown status";
  }
}

int fd_version(void) { return (0 << 16) | (1 << 8) | 0; }

}  // extern "C"
