// Declarations shared by the library's translation units (not part of the C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Device-side status word, one per device. A kernel that gives up a bounded
// wait writes its code here (first writer wins) and exits; fa_last_status()
// reads and clears it after synchronising.
struct DevStatus {
  unsigned int code;    // 0 = ok, kStatusTimeout, ...
  unsigned int kernel;  // KernelId of the first failing kernel
  unsigned int site;    // which wait inside that kernel
  unsigned int block;   // linear block index
};
constexpr unsigned int kStatusTimeout = 4u;  // matches FA_ERR_TIMEOUT

enum KernelId : unsigned int {
  kKernFwd = 1,
  kKernFwdF32 = 2,
  kKernBwdDelta = 3,
  kKernBwdDkDv = 4,
  kKernBwdDq = 5,
  kKernDecodeSplit = 6,
  kKernDecodeCombine = 7,
  kKernFwdFp8 = 8,
};

// Numeric storage types, same values as the C ABI's fa_dtype; kU8 (bytes: the FP8 path's E4M3
// operands) is internal.
enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2, kU8 = 3 };

inline size_t dtype_size(int dt) { return dt == kF32 ? 4u : 2u; }

// Test-only fault injections (fa_debug_inject): which launch they reach and what it skips.
constexpr int kInjectDecodeStage = 1;  // decode: CTA 0 never loads its first stage of keys
constexpr int kInjectFwdStage = 2;     // D = 64 forward: CTA 0 never loads its first K/V stage
constexpr int kInjectFwdFlag = 3;      // D = 64 forward, split schedule: CTA 1 never publishes its partial
constexpr int kInjectBwdCount = 4;     // fused backward, split schedule: the first CTA holding a later
                                       // piece of a cut key tile never counts its partial in

// Per-launch context every kernel receives.
struct LaunchCtx {
  DevStatus* status;
  unsigned long long wait_budget_ns;
  int num_sms;
  cudaStream_t stream;
  int inject = 0;  // test-only fault injection for this launch (see fa_debug_inject)
};

// ---- launchers (each returns a cudaError_t from the launch itself)
// Decode: `rows` (1..kDecMaxRows) query rows per (batch, head); LSE may be null.
constexpr int kDecMaxRows = 4;
cudaError_t launch_decode(const void* q, const void* K, const void* V, void* O, float* LSE, float* ws, int BH,
                          int rows, int N, int D, float scale, int n_splits, int dtype, const LaunchCtx& ctx);

// Split schedule of the D = 64 forward: the caller's workspace holds one
// partial-result slot and 8 ready flags per SM; ws == nullptr selects the classic schedule.
// epoch is unique per launch (flags from earlier launches never match it).
struct FwdSplit {
  float* ws = nullptr;
  uint32_t* flags = nullptr;
  uint32_t epoch = 0;
};
size_t fwd_d64_split_bytes(int num_sms);
// head dimension 64 only (fp16 / bf16); called by launch_fwd_half
cudaError_t launch_fwd_d64(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M, int N,
                           float scale, bool causal, int dtype, const FwdSplit& sp, const LaunchCtx& ctx);
cudaError_t launch_fwd_half(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M, int N,
                            int D, float scale, bool causal, int dtype, const FwdSplit& sp, const LaunchCtx& ctx);

// f32 forward; with few query tiles (under half the SMs) each tile's key blocks are shared by
// `parts` CTAs, and the one that finishes last merges the others' partials (ws:
// fwd_f32_split_bytes bytes of partial slots and per-tile counters; epoch: nonzero, new per
// launch, so counts an earlier launch left behind read as zero).
int fwd_f32_parts(int BH, int M, int N, int num_sms);
size_t fwd_f32_split_bytes(int BH, int M, int parts);
constexpr int kF32SlotFloats = 64 * 128 + 2 * 128;  // one part's partial: O [64][128 rows], m, l
// The f32 forward with a workspace (D = 64): a prologue kernel writes K's tf32 hi and lo parts and
// V's transposed hi and lo parts into `presplit` (fwd_f32_presplit_bytes), then the main kernel
// streams them (split_ws, parts, epoch as for launch_fwd_f32).
size_t fwd_f32_presplit_bytes(int BH, int N);
cudaError_t launch_fwd_f32_presplit(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M,
                                    int N, float scale, bool causal, int parts, float* split_ws, uint32_t epoch,
                                    void* presplit, const LaunchCtx& ctx);
cudaError_t launch_fwd_f32(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH, int M, int N,
                           int D, float scale, bool causal, int parts, float* ws, uint32_t epoch,
                           const LaunchCtx& ctx);

// The FP8 forward's workspace (head dimension 64): E4M3 copies of Q [BH][M][64] and K
// [BH][N][64] after the Hadamard-times-sign transform, V transposed [BH][64][npad] (npad = N
// rounded up to 16), the per-block scales sq [BH][ceil(M/128)] and sk [BH][ceil(N/128)], V's
// per-block maxima vmax [BH][ceil(N/128)] and per-head scale sv [BH].
struct Fp8Ws {
  uint8_t *q8, *k8, *vt8;
  float *sq, *sk, *vmax, *sv;
  int npad;
};
cudaError_t launch_fp8_quant(const void* Q, const void* K, const void* V, const int8_t* signs, const Fp8Ws& w, int BH,
                             int M, int N, int dtype, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const Fp8Ws& w, void* O, float* LSE, int BH, int M, int N, float scale, bool causal,
                           int dtype, const LaunchCtx& ctx);

// Split schedule of the fused backward (non-causal, D = 64): ws holds bwd_fused_split_bytes of
// partial dK/dV slots (two per SM) then num_sms * 8 counters; ws == nullptr runs whole key tiles.
struct BwdSplit {
  float* ws = nullptr;
  bool pair = false;  // three-kernel path, D = 64: the dK/dV and dQ kernels on CTA pairs
};
size_t bwd_fused_split_bytes(int num_sms);

// dK / dV with D = 64 on CTA pairs (cta_group::2), launched as a programmatic dependent of the
// delta kernel; the three-kernel backward's alternative to its single-CTA dK/dV kernel.
cudaError_t launch_bwd_dkdv64_pair(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                                   const float* delta, void* dK, void* dV, int BH, int M, int N, float scale,
                                   bool causal, int dtype, const LaunchCtx& ctx);
// dQ with D = 64 on CTA pairs, launched as a programmatic dependent of the dK/dV kernel.
cudaError_t launch_bwd_dq64_pair(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                                 const float* delta, void* dQ, int BH, int M, int N, float scale, bool causal,
                                 int dtype, const LaunchCtx& ctx);

// dQacc == nullptr: delta, dK/dV and dQ kernels; else (D = 64) delta, one fused dK/dV/dQ kernel
// that accumulates dQ in dQacc (B*H*M*D f32), and a conversion of dQacc into dQ.
cudaError_t launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, float* delta, float* dQacc, int BH, int M, int N, int D,
                       float scale, bool causal, int dtype, const BwdSplit& sp, const LaunchCtx& ctx);

// Entry-point helpers of fa_api.cu used by the other host translation units: the decode
// entry points' checks and launch, and recording a failure's one-line reason.
fa_status decode_entry(const void* q, const void* Kcache, const void* Vcache, void* O, float* LSE, float* partial_ws,
                       int B, int H, int R, int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream,
                       const char* name);
fa_status fail_msg(fa_status s, const char* msg);
fa_status cuda_fail_msg(cudaError_t e, const char* what);

// Encodes a 3-D TMA tensor map over a contiguous [outer, rows, inner] tensor
// (inner = head dimension) with a box of [box_inner, box_rows, 1] elements and
// 128-byte swizzle. Returns false when the driver rejects it.

bool make_tmap_3d(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows, uint64_t outer,
                  uint32_t box_inner, uint32_t box_rows);
// The same with the swizzle span chosen: 128 or 64 bytes (the box's inner extent in bytes
// must not exceed it).
bool make_tmap_3d_ex(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows, uint64_t outer,
                     uint32_t box_inner, uint32_t box_rows, int swizzle_bytes);
// A view of the first `inner` elements of rows `pitch` elements apart (128-byte swizzle); a box
// wider than the view reads the columns past it as zeros. False when the driver refuses it.
bool make_tmap_3d_view(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t pitch, uint64_t rows,
                       uint64_t outer, uint32_t box_inner, uint32_t box_rows);

}  // namespace fa
