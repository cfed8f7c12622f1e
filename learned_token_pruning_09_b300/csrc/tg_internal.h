// Internal declarations shared by the C-ABI layer (tg_api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace tg {

// device status codes (same values as tg_status)
constexpr unsigned int kStatusTimeout = 5;
constexpr unsigned int kStatusIndex = 6;

constexpr int kMaxHeadDimHalf = 64;

struct RopeFreqs {
  // theta^(-2i/D) / (2 pi), i < D/2, in turns per position, as hi + lo fp32
  float turns_hi[kMaxHeadDimHalf];
  float turns_lo[kMaxHeadDimHalf];
};

// ---- score histograms of the top-K workspace ------------------------------
// Per sequence: kHistCoarse counts of the top 8 bits of the scores' order
// keys, then kHistFine counts of their top 16 bits, bin f stored at
// fine_slot(f): scores cluster in a few hundred consecutive bins, and
// transposing the two bytes puts those bins 1 KB apart, on many L2 slices,
// instead of on a handful of cache lines that the gate's atomics would queue
// on (slowing the residual stream through the same slices).
constexpr int kHistCoarse = 256;
constexpr int kHistFine = 65536;
__host__ __device__ constexpr uint32_t fine_slot(uint32_t f) { return ((f & 255u) << 8) | (f >> 8); }
constexpr int kHistWords = kHistCoarse + kHistFine;
constexpr int kTopkMaxHistBatch = 65535;   // the gate packs (sequence, 16-bit bin) into 32 bits

// ---- gate ------------------------------------------------------------------
struct GateArgs {
  uint32_t* hist;           // [batch][kHistWords] score histograms to add to, or null
  const uint8_t* prunable;  // [n_rows] per-row mask, or null: the document prefix (n_doc)
  const float* b1;          // [h] or null
  const __nv_bfloat16* w2;  // [h]
  float b2;
  const int32_t* cu_seqlens;
  const int32_t* n_doc;
  int32_t batch;
  int64_t n_rows;
  int32_t d;
  int32_t h;
  float* s_out;
  unsigned int* status;
  long long watchdog;
  int num_sms;
};
cudaError_t launch_gate(const CUtensorMap& map_x, const CUtensorMap& map_w1, const GateArgs& a,
                        cudaStream_t st);

// ---- top-K -----------------------------------------------------------------
struct TopkArgs {
  uint32_t* hist;           // [batch][kHistWords] the gate's score histograms (zeroed after use), or null
  const float* s;
  const int32_t* cu_seqlens;
  // Prunable rows of each sequence: with `prunable` null, the first n_doc[b]
  // rows (the document) and the rest (the question) always kept; with a
  // per-row mask, the masked rows, n_doc[b] of them (counted by
  // launch_topk_count first), anywhere in the sequence.
  const int32_t* n_doc;
  const uint8_t* prunable;
  const int32_t* k;
  int32_t batch;
  int32_t max_n_doc;        // host bound on the rows a sequence's slices cover
  int64_t kept_capacity;    // length of kept_idx
  int32_t* kept_idx;
  int32_t* cu_kept;
  unsigned int* status;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st);
// n_prun[b] = number of prunable rows of sequence b
cudaError_t launch_topk_count(const uint8_t* prunable, const int32_t* cu_seqlens, int32_t batch,
                              int32_t* n_prun, unsigned int* status, cudaStream_t st);

// ---- gather ----------------------------------------------------------------
struct GatherArgs {
  const void* x;
  int64_t n_rows;           // rows of x (and s)
  int32_t d;
  const float* s;
  const int32_t* cu_seqlens;
  const int32_t* kept_idx;
  const int32_t* cu_kept;
  int32_t batch;
  int64_t n_kept;
  void* x_kept;
  int32_t* pos_kept;
  float* s_kept;
  unsigned int* status;
  long long watchdog;
  int num_sms;
};
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t st);

// ---- RoPE prologue ---------------------------------------------------------
struct RopeArgs {
  const void* q;        // [T, hq, D]
  const void* k;        // [T, hkv, D]
  const int32_t* pos;   // [T]
  const int32_t* cu_kept;
  int32_t batch;
  int64_t n_kept;
  int32_t hq, hkv, head_dim;
  void* q_out;
  void* k_out;
  unsigned int* status;
  int num_sms;
};
cudaError_t launch_rope(const RopeArgs& a, const RopeFreqs& f, cudaStream_t st);

// ---- attention -------------------------------------------------------------
struct AttnArgs {
  const int32_t* pos;
  const float* s_kept;
  const float* gain;
  const int32_t* cu_kept;
  int32_t batch;
  int64_t n_kept;
  int32_t max_kept;
  int32_t hq, hkv, head_dim;
  float scale_log2;     // log2(e) / (sqrt(D) * tau)
  float bias_unit;      // sqrt(D) * tau: the score bias in units of q.k
  void* o;
  float* lse;
  unsigned int* status;
  long long watchdog;
};
cudaError_t launch_attention(const CUtensorMap& map_q, const CUtensorMap& map_k,
                             const CUtensorMap& map_v, const AttnArgs& a, cudaStream_t st);

// ---- attention backward: gradients of the score, gain and temperature ------
constexpr int kBwdMaxGroup = 8;   // query heads per KV head
constexpr int kBwdChunks = 32;    // key chunks per head in the dgain / dtau reduction
constexpr int kBwdMaxHeads = 256; // query heads (the final reduction holds one per thread)
struct AttnBwdArgs {
  const void* o;          // [T, hq, D] bf16, the forward output
  const void* d_o;        // [T, hq, D] bf16
  const float* lse;       // [hq, T] natural log, from the forward
  const int32_t* pos;
  const float* s_kept;
  const float* gain;
  const int32_t* cu_kept;
  int32_t batch;
  int64_t n_kept;
  int32_t max_kept;
  int32_t hq, hkv, head_dim;
  float scale_log2;       // log2(e) / (sqrt(D) tau)
  float dtau_scale;       // -1 / (sqrt(D) tau^2)
  float* delta;           // [hq, T] workspace: dO_i . o_i
  float* r_part;          // [2, hq, T] workspace: sum_i dl_ij, per softmax warpgroup
  float* t_part;          // [2, hq, T] workspace: sum_i dl_ij (q'_i . k'_j), per warpgroup
  float* part;            // [hq, kBwdChunks, 2] workspace: per-chunk sums for dgain and dtau
  float* ds;              // [T]
  float* dgain;           // [hq]
  float* dtau;            // [1]
  unsigned int* status;
  long long watchdog;
  int num_sms;
};
cudaError_t launch_attention_bwd(const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                                 const CUtensorMap& map_do, const AttnBwdArgs& a, cudaStream_t st);

// ---- pruned Gated DeltaNet scan --------------------------------------------
struct ScanArgs {
  const void* q;              // [T, hk, dk] bf16
  const void* k;              // [T, hk, dk] bf16
  const void* v;              // [T, hv, dv] bf16
  const float* g;             // [T, hv] log-decays
  const float* beta;          // [T, hv]
  const int32_t* cu_kept;
  int32_t batch;
  int64_t n_kept;
  int32_t hk, hv, dk, dv;
  float scale;
  const float* initial_state; // [batch, hv, dv, dk] or null (zero)
  void* o;                    // [T, hv, dv] bf16
  float* final_state;         // [batch, hv, dv, dk] or null
  unsigned int* status;
  void* ws;                   // chunked form: per-chunk products (delta_chunked_ws_bytes), or null
  long long watchdog;
  int num_sms;
};
cudaError_t launch_delta_scan(const ScanArgs& a, cudaStream_t st);
// chunked form on the tensor cores (dk 64 or 128, dv <= 128), with a workspace
cudaError_t launch_delta_scan_chunked(const ScanArgs& a, cudaStream_t st);
size_t delta_chunked_ws_bytes(long long n_kept, int batch, int hv, int dk, int dv);

// ---- the layer around the pruned path: norms, SwiGLU, decode attention -----
cudaError_t launch_rms_norm(const void* x, const void* w, long long rows, int d, float eps, void* y, int num_sms,
                            cudaStream_t st);
cudaError_t launch_swiglu(const void* gate_up, long long rows, int f, void* y, int num_sms, cudaStream_t st);
constexpr int kDecodeMaxGroup = 8;   // query heads per KV head
constexpr int kDecodeSplit = 256;    // cache rows per CTA
struct DecodeArgs {
  const void* q;          // [B, hq, D] bf16, rotated
  const void* k_new;      // [B, hkv, D] bf16, rotated
  const void* v_new;      // [B, hkv, D] bf16
  const void* k_cache;    // [cache_rows, hkv, D] bf16, rotated
  const void* v_cache;    // [cache_rows, hkv, D] bf16
  const int32_t* cache_cu;
  const float* s_cache;   // [cache_rows] or null (no score bias)
  const float* gain;      // [hq] or null
  int32_t batch;
  int64_t cache_rows;
  int32_t hq, hkv, head_dim;
  int32_t split_len, n_split;
  float scale_log2;       // log2(e) / (sqrt(D) tau)
  float* part;            // [B, hq, n_split, D + 2] workspace
  void* o;                // [B, hq, D] bf16
  unsigned int* status;
};
cudaError_t launch_decode_attention(const DecodeArgs& a, cudaStream_t st);

// ---- linear ----------------------------------------------------------------
struct LinearArgs {
  const void* residual;
  void* out;
  int64_t m;
  int32_t n;
  int32_t kdim;
  unsigned int* status;
  long long watchdog;
  int num_sms;
  // Q/K/V projection with RoPE (out == null): the columns form heads of
  // head_dim; the first hq heads go to q_out [m, hq, D], the next hkv to
  // k_out [m, hkv, D], the rest to v_out [m, hkv, D]; q and k heads are
  // rotated at pos[row]
  void* q_out;
  void* k_out;
  void* v_out;
  const int32_t* pos;
  int32_t hq, hkv, head_dim;
  RopeFreqs freqs;
};
// Columns of a linear tile: 256, or n itself when smaller (n is a multiple
// of 16, so each CTA of a pair stages a multiple of 8 rows of W).
inline int linear_tile_n(int n) { return n >= 256 ? 256 : n; }
cudaError_t launch_linear(const CUtensorMap& map_a, const CUtensorMap& map_w, const LinearArgs& a,
                          cudaStream_t st);

}  // namespace tg
