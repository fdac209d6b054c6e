// Internal interface between the host API (fd_api.cpp) and the kernels
// (fd_kernels.cu). Not installed; the public interface is
// include/fd_decode_attn.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace fd {

// Everything a launch needs; filled and validated by the host API.
struct LaunchArgs {
  const uint16_t* q;        // bf16 [B][NH][HS]
  const uint16_t* k;        // bf16 [B][NKV][capacity][HS]
  const uint16_t* v;        // bf16 [B][NKV][capacity][HS]
  uint16_t* out;            // bf16 [B][NH][HS]
  float* out_f32;           // fp32 [B][NH][HS] or nullptr
  const int* lens;          // int32 [B]
  float* ws_o;              // fp32 [B][NH][S][HS]  (S > 1 only)
  float* ws_ml;             // fp32 [B][NH][S][2]   (m in log2 units, l)
  unsigned int* counters;   // [B][NKV] finished-split counters (fused merge), zero between calls;
                            // with the group step, [B][NKV] count-out words after them
  unsigned int* work_counter;  // persistent grid: next work item, zero between calls
  int persistent;           // blocks of a persistent split grid; 0: one block per split
  int fused;                // 1: the last split block of each (b, kvh) merges; 2: every split block
                            // of a group waits for the group, then merges a share; no merge kernel
  int group_bytes;          // bytes per bulk-copy group of the tile (2048, or 4096 for the wide MQA tile)
  int consumer_warps;       // consumer warps of the split tile (the plan's choice)
  int kv8;                  // 1: the cache is E4M3 codes (k8/v8) with per-(b, kvh) scales
  const uint8_t* k8;        // E4M3 [B][NKV][capacity][HS]  (kv8 only)
  const uint8_t* v8;        // E4M3 [B][NKV][capacity][HS]  (kv8 only)
  const float* k_scale;     // fp32 [B][NKV]                 (kv8 only)
  const float* v_scale;     // fp32 [B][NKV]                 (kv8 only)
  int B, NH, NKV, HS, capacity, window;  // window <= 0: none
  int num_splits;           // S
  int cluster;              // blocks per cluster along the splits (S % cluster == 0)
  int granule;              // chunk rounding, positions
  int tile_stride;          // > 0: the split kernel dealt T = tile_stride position tiles to the splits in
                            // turn (bands of slots [0, band)); 0: consecutive chunks (set at launch)
  int path;                 // FD_PATH_SIMT / FD_PATH_TC / FD_PATH_UMMA
  int min_len;              // every lens[b] >= min_len (the caller's bound; 0: none): tiles of slots
                            // [0, min(min_len, capacity)) are live before the lengths are read
  int withhold_tile;        // test hook: tensor-core split blocks issue no copies from this tile of
                            // theirs on (a huge value: off)
  int one_tile;             // 1: the plan gives every split at most one tile (whole-tile splits
                            // covering its band bound), so a one-stage tile may serve it
  float scale_log2;         // scale * log2(e)
};

// Positions per pipeline tile of the tensor-core kernel for head size HS, and
// the chunk granule the plan uses for it.
int tc_tile_positions(int HS, bool kv8);
// Positions of the short-band E4M3 tile (1 KB groups) for head sizes 64 and
// 128; 0 for the others.
int tc_short_tile_positions(int HS);
int plan_granule(int path, int HS, bool kv8);

// Resident CTAs per SM of the kernel a plan would launch (occupancy query).
cudaError_t query_ctas_per_sm(int path, int HS, int G, bool kv8, int* ctas);

// Largest cluster size (16, 8, ... 1) of the tensor-core split kernel that the
// device can schedule (cluster occupancy query).
cudaError_t query_max_cluster(int HS, int G, bool kv8, int* cluster);

// The tcgen05 / tensor-memory split kernel (fd_umma.cu): bf16, head dim 512,
// 8 < G <= 16 query rows per KV head, no window.
bool umma_shape_ok(int HS, int G, int window);
int umma_tile_positions();
cudaError_t launch_umma(const LaunchArgs& a, cudaStream_t stream);
cudaError_t read_and_clear_device_error_umma(unsigned int* err);

// Launch the split kernel (and the merge kernel when S > 1) on `stream`.
cudaError_t launch_decode(const LaunchArgs& a, cudaStream_t stream);

// Read and clear the device error word of the current device.
cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* err);

// Wall-time limit of the kernels' bounded waits on the current device, in
// nanoseconds (0: the default, about one second); one setter per
// translation unit that holds kernels.
cudaError_t set_wait_limit(unsigned long long ns);
cudaError_t set_wait_limit_umma(unsigned long long ns);

// fd_decode_attn_noalloc (fd_noalloc.cu): forget each device's scratch set-up,
// so the next call clears the scratch again.
void noalloc_forget();

}  // namespace fd
