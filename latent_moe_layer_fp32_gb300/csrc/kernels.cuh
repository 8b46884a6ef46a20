// Kernel declarations and launch-side configuration shared by the .cu files.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace lmoe {

// ---- api.cu: argument checks and launch bookkeeping shared by the entry points ----
// LMOE_OK, LMOE_EINVAL or LMOE_EUNSUPPORTED for the layer dimensions
int check_dims(const lmoe_dims* d);
// split-K factor of the CUDA-core router: enough CTAs for the GPU, at most max_split
int router_splits(int T, int E, int H, int sms, int max_split);
// K range per warp of route_fast_kernel (at most 16 ranges), or 0 when H does not allow it
int fast_route_ks(int H);
// per-call launch count and names (lmoe_last_launch_count / _name) and the optional
// per-launch timing events (lmoe_profile_events)
void calls_begin();
void pre_launch(cudaStream_t s, const char* name);
void launched();

// ---- route.cu -------------------------------------------------------------
// g (optional): the sandwich block's pre-norm gain, the router input becomes x * g;
// rinv (optional): per-token scale of the summed dot products (before the bias)
__global__ void router_partial_kernel(const uint16_t* x, const float* wr, float* part, int T, int H, int E,
                                      int split_len, const uint16_t* g);
__global__ void topk_kernel(const float* part, int nsplit, const float* bias, int T, int E, int k,
                            int32_t* topk_idx, float* topk_w, const float* rinv);
__global__ void route_small_kernel(const uint16_t* x, const float* wr, const float* bias, float* part, int T, int H,
                                   int E, int k, int split_len, int G, int32_t* topk_idx, float* topk_w,
                                   int32_t* offsets, int32_t* sorted_rows, int32_t* row_pos, int4* groups,
                                   int32_t* n_groups, int32_t* tickets, Status* st, const uint16_t* g,
                                   const float* rinv);
__global__ void route_fast_kernel(const uint16_t* x, const float* wr, const float* bias, float* part, int T, int H,
                                  int E, int k, int KS, int G, int32_t* topk_idx, float* topk_w, int32_t* offsets,
                                  int32_t* sorted_rows, int32_t* row_pos, int4* groups, int32_t* n_groups,
                                  int32_t* tickets, Status* st, const uint16_t* g, const float* rinv);
__global__ void router_split_kernel(const float* wr, int E, int H, uint16_t* w3, int dup);
constexpr int kChunkTok = 32;  // tokens per chunk of the many-token routing table
__global__ void topk_hist_kernel(const float* part, int nsplit, const float* bias, int T, int E, int k,
                                 int32_t* topk_idx, float* topk_w, int32_t* rank, int32_t* chunk_cnt,
                                 const float* rinv);
__global__ void table_hist_kernel(const int32_t* topk_idx, int T, int E, int k, int32_t* rank, int32_t* chunk_cnt,
                                  Status* st);
__global__ void table_scan_kernel(int32_t* chunk_cnt, int nchunks, int E, int R, int G, int32_t* offsets,
                                  int4* groups, int32_t* n_groups);
__global__ void table_scatter_kernel(const int32_t* topk_idx, const int32_t* rank, const int32_t* chunk_base, int R,
                                     int E, int k, int32_t* sorted_rows, int32_t* row_pos);
__global__ void table_kernel(const int32_t* topk_idx, int R, int E, int G, int32_t* offsets, int32_t* sorted_rows,
                             int32_t* row_pos, int4* groups, int32_t* n_groups, Status* st);

// ---- experts.cu -----------------------------------------------------------
// Group of up to G rows (sorted positions p0 .. p0+n-1) of one expert e:
// int4 {e, p0, n, 0}.
struct ExpertArgs {
  const uint8_t* q;         // codes [E][rows_per_expert][K/2]
  const uint8_t* s;         // scales [E][rows_per_expert][K/32] E8M0, or [K/16] E4M3 when gs is set
  const float* gs;          // NVFP4: fp32 global scale per expert matrix [E]; null for MXFP4
  const uint16_t* act;      // bf16 activations, row-major [*][K] (x_lat by token, or h by sorted position)
  const int4* groups;       // group list
  const int32_t* n_groups;  // device count of groups
  const int32_t* sorted_rows;
  int K;                    // reduction width (L for gate/up, I for down)
  int kc;                   // K chunk per stage
  int inter;                // I
  int latent;               // L
  int top_k;
  int n_experts;
  uint16_t* h_out;          // gate/up: bf16 [R_sorted][I]
  float* y_out;             // down: fp32 [R][L] by original row id
  float* ssq_out;           // down: fp32 [R][L/32] sum of y^2 per 32-row tile (may be null)
  Status* st;
  int groups_cap;           // entries allocated in groups (read ahead speculatively up to this)
  int rows;                 // R = T * k: entries of sorted_rows
  int early;                // 1: the group list comes from a kernel before the preceding one, so the
                            // first weights stream before the programmatic-launch wait; 0: wait first
  // down only, at most 64 route rows: the post-expert norm and the weighted sum
  // in the same launch (after a device-wide count of the CTAs done), else null
  uint16_t* zb;             // bf16 [T][L] z
  const int32_t* topk_idx;  // [T][k]
  const float* topk_w;      // [T][k]
  const uint16_t* norm_g;   // bf16 [E][L]
  int32_t* zctr;            // zeroed before the launch
  float eps;
  int T;
};

int launch_gateup(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms);
int launch_down(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms);
int expert_max_group(int T);

// ---- fused_experts.cu ------------------------------------------------------
// Decode-size experts (T <= 8, T*k <= 64 route rows), MXFP4: gate/up + SwiGLU
// and down in one persistent launch (one CTA per SM, a device-wide counter
// between the two stages).
struct FusedExpertArgs {
  const uint8_t* w13_q;     // [E][2I][L/2]
  const uint8_t* w13_s;     // [E][2I][L/32]
  const uint8_t* w2_q;      // [E][L][I/2]
  const uint8_t* w2_s;      // [E][L][I/32]
  const uint16_t* x_lat;    // bf16 [T][L]
  const int4* groups;       // group list {e, p0, n, 0}
  const int32_t* n_groups;
  const int32_t* sorted_rows;
  uint16_t* h;              // bf16 [R][I] by sorted position (written, then read back)
  uint16_t* h_out;          // = h
  float* y_out;             // fp32 [R][L] by original row id
  float* ssq_out;           // fp32 [R][L/32]
  int32_t* ctr;             // [65] zero at launch: per-group counts of finished gate/up items, then
                            // the number of CTAs done with their down items
  Status* st;
  // the layer's norm and weighted sum (null zb: the experts alone)
  const int32_t* topk_idx;  // [T][k]
  const float* topk_w;      // [T][k]
  const uint16_t* norm_g;   // bf16 [E][L]
  uint16_t* zb;             // out bf16 [T][L]
  float eps;
  int T, latent, inter, top_k, n_experts, rows;
  int early;                // 1: the routing table was written before the preceding kernel ran
};
int launch_fused_experts(const FusedExpertArgs& a, cudaStream_t s, int num_sms);

// ---- gemv.cu --------------------------------------------------------------
// When the kernel waits for the preceding kernel of the stream (programmatic
// dependent launch): before anything (0); after issuing the weight copies of its
// first ring slots, which depend on nothing earlier (1); at its very end, the
// whole projection depending on nothing earlier in the stream (2).
enum { kWaitFirst = 0, kWaitAfterWeights = 1, kWaitAtEnd = 2 };

struct GemvArgs {
  const uint16_t* w;    // bf16 [N][K]
  const uint16_t* act;  // bf16 [T][K]
  uint16_t* out;        // bf16 [T][N]
  int N, K, T;
  Status* st;
  int wait_mode;        // kWaitFirst, kWaitAfterWeights or kWaitAtEnd
};
int launch_gemv_bf16(const GemvArgs& a, cudaStream_t s, int num_sms);

// ---- tc_gemm.cu -----------------------------------------------------------
// out[M][N] = bf16_rne(A[M][K] . B[N][K]^T) on tcgen05; N % 256 == 0, K % 64 == 0,
// A, B, out 16-byte aligned.
struct TcGemmArgs {
  uint16_t* out;        // bf16 [M][N] (unless out_f32 is set)
  int M, N, K;
  Status* st;
  float* out_f32;       // optional: fp32 partial sums [nsplit][M][N] instead of bf16 out
  int a_kblocks;        // > 0: A's 64-wide k-block index wraps modulo this (A reused along K)
  int n_tile;           // output columns per tile: 256 (0), or a multiple of 32 below it
  int nsplit;           // K split into this many ranges, one partial each (0 or 1: none)
  // optional (bf16 output only): also write output row m to rows scatter_pos[m*scatter_k + j]
  // (j < scatter_k) of scatter_out [*][N] -- x_lat rows in expert-sorted order for the experts
  const int32_t* scatter_pos;
  int scatter_k;
  uint16_t* scatter_out;
};
int launch_tc_gemm_bf16(const TcGemmArgs& a, const uint16_t* A, const uint16_t* B, cudaStream_t s, int num_sms);
constexpr int kTcGemmN = 256, kTcGemmK = 64;

// ---- tc_experts.cu ---------------------------------------------------------
// Grouped W4A16 expert GEMMs on tcgen05 (groups of up to 256 sorted rows).
struct TcExpertArgs {
  const uint8_t* q;         // codes [E][rows_per_expert][K/2]
  const uint8_t* s;         // scales [E][rows_per_expert][K/32] E8M0, or [K/16] E4M3 when gs is set
  const float* gs;          // NVFP4: fp32 global scale per expert matrix [E]; null for MXFP4
  const int4* groups;       // {e, p0, n <= 256, 0}
  const int32_t* n_groups;
  const int32_t* sorted_rows;  // down: original row id of each sorted position
  int K;                    // L (gate/up) or I (down)
  int inter, latent, n_experts;
  int rows;                 // R = T * k
  uint16_t* h_out;          // gate/up: bf16 [R][I] by sorted position
  float* y_out;             // down: fp32 [R][L] by original row id
  float* ssq_out;           // down: fp32 [R][L/32] sum of y^2 per 32-column tile
  Status* st;
};
int launch_tc_gateup(const TcExpertArgs& a, const uint16_t* x_sorted, cudaStream_t s, int num_sms);
int launch_tc_down(const TcExpertArgs& a, const uint16_t* h, cudaStream_t s, int num_sms);
constexpr int kTcExpertGroup = 160;
__global__ void gather_rows_kernel(const uint16_t* x_lat, const int32_t* sorted_rows, int R, int k, int L,
                                   uint16_t* x_sorted);
__global__ void dequant_selftest_kernel(const uint8_t* codes, const uint8_t* scales, int nblocks, uint16_t* out);

// ---- misc.cu --------------------------------------------------------------
__global__ void groups_from_offsets_kernel(const int32_t* offsets, const int32_t* sorted_rows, int E, int R, int G,
                                           int4* groups, int32_t* n_groups, Status* st);
__global__ void ssq_kernel(const float* y, int R, int L, float* ssq);
__global__ void ws_zero_kernel(uint4* p, int n16);
__global__ void io_in_kernel(const uint4* x_host, uint4* x_dev, size_t n16, uint4* zero, int nzero16);
__global__ void io_out_kernel(const uint4* out_dev, uint4* out_host, size_t n16);
__global__ void timeout_selftest_kernel(Status* st, unsigned long long limit_ns);
// ---- block.cu -------------------------------------------------------------
__global__ void prenorm_kernel(const uint16_t* x, const uint16_t* g, float eps, int H, uint16_t* n_bf16, float* rinv,
                               uint16_t* u_split);
__global__ void postnorm_residual_kernel(const uint16_t* out, const uint16_t* x, const uint16_t* g, float eps, int H,
                                         uint16_t* y);

__global__ void combine_kernel(const float* y, const float* ssq, const int32_t* topk_idx, const float* topk_w,
                               const uint16_t* norm_g, int L, int k, int E, float eps, uint16_t* zb, Status* st);
__global__ void e2m1_selftest_kernel(float* out);

}  // namespace lmoe
