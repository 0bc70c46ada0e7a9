// The C ABI of libfa: argument checks, per-device state, TMA descriptor
// encoding and dispatch to the kernel launchers. See include/fa.h for the
// contract of each entry point.
#include <cudaTypedefs.h>

#include <cinttypes>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <algorithm>
#include <chrono>
#include <cmath>
#include <mutex>
#include <vector>

#include "../../include/fa.h"
#include "fa_internal.cuh"

namespace fa {

__device__ DevStatus g_status;  // one per device that loads the library

namespace {

constexpr int kMaxDevices = 64;

struct DevState {
  bool ready = false;
  int num_sms = 0;
  DevStatus* status = nullptr;  // device address of g_status on this device
};

std::mutex g_mutex;
DevState g_dev[kMaxDevices];
unsigned long long g_wait_budget_ns = 0;  // 0 = not yet read from the environment
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local char t_msg[512] = "";

fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

unsigned long long wait_budget() {
  if (g_wait_budget_ns == 0) {
    unsigned long long v = 2000000000ull;
    if (const char* e = std::getenv("FA_WAIT_BUDGET_NS")) {
      unsigned long long x = std::strtoull(e, nullptr, 10);
      if (x >= 1000ull) v = x;
    }
    g_wait_budget_ns = v;
  }
  return g_wait_budget_ns;
}

// Per-device set-up, done once with that device current: SM count and the
// device address of the status word.
fa_status device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  DevState& st = g_dev[dev];
  if (!st.ready) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    DevStatus zero{};
    e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    st.num_sms = sms;
    st.status = static_cast<DevStatus*>(p);
    st.ready = true;
  }
  wait_budget();
  *out = &st;
  return FA_OK;
}

fa_status make_ctx(LaunchCtx* ctx, void* stream) {
  DevState* st = nullptr;
  fa_status s = device_state(&st);
  if (s != FA_OK) return s;
  ctx->status = st->status;
  ctx->num_sms = st->num_sms;
  ctx->wait_budget_ns = wait_budget();
  ctx->stream = static_cast<cudaStream_t>(stream);
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_dtype(int dtype) {
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return fail(FA_ERR_INVALID, "unknown dtype %d", dtype);
  return FA_OK;
}

fa_status check_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(FA_ERR_INVALID, "%s is NULL", name);
  if (!aligned16(p)) return fail(FA_ERR_INVALID, "%s is not 16-byte aligned", name);
  return FA_OK;
}

// Rejects element counts whose byte size or whose row index would overflow the
// 32-bit row coordinates the kernels and TMA descriptors use.
fa_status check_sizes(int B, int H, int M, int N, int D) {
  if (B < 0 || H < 0 || M < 0 || N < 0 || D <= 0)
    return fail(FA_ERR_INVALID, "negative or zero size (B=%d H=%d M=%d N=%d D=%d)", B, H, M, N, D);
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT_MAX) return fail(FA_ERR_INVALID, "B*H overflows int");
  if (bh * static_cast<long long>(M > N ? M : N) > static_cast<long long>(INT_MAX))
    return fail(FA_ERR_INVALID, "B*H*max(M,N) = %lld rows overflows int", bh * (M > N ? M : N));
  if (D != 64 && D != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension D=%d (supported: 64, 128)", D);
  return FA_OK;
}

// Any finite scale: the tensor-core paths negate the score product in the tensor core when
// scale < 0 and scale the exponent by |scale|.
fa_status check_scale(float scale) {
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(FA_ERR_INVALID, "scale must be finite (got %g)", static_cast<double>(scale));
  return FA_OK;
}

#define FA_TRY(expr)                 \
  do {                               \
    fa_status _s = (expr);           \
    if (_s != FA_OK) return _s;      \
  } while (0)

}  // namespace

bool make_tmap_3d(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows, uint64_t outer,
                  uint32_t box_inner, uint32_t box_rows) {
  return make_tmap_3d_ex(map, base, dtype, inner, rows, outer, box_inner, box_rows, 128);
}

bool make_tmap_3d_ex(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows, uint64_t outer,
                     uint32_t box_inner, uint32_t box_rows, int swizzle_bytes) {
  if (g_encode == nullptr) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const size_t es = dtype == kU8 ? 1u : dtype_size(dtype);
  CUtensorMapDataType t = dtype == kF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                          : dtype == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                          : dtype == kU8  ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * es, inner * rows * es};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_3d_view(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t pitch, uint64_t rows,
                       uint64_t outer, uint32_t box_inner, uint32_t box_rows) {
  if (!make_tmap_3d(map, base, dtype, pitch, rows, outer, box_inner, box_rows)) return false;  // loads the encoder
  const size_t es = dtype_size(dtype);
  const CUtensorMapDataType t = dtype == kF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : dtype == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {pitch * es, pitch * rows * es};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa

using namespace fa;

namespace {

size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

// Schedule choices fixed by fa_set_schedule (-1: automatic). Process-wide.
std::atomic<int> g_sched_fwd_split{-1};
std::atomic<int> g_sched_bwd_split{-1};
std::atomic<int> g_sched_host_chunks{-1};
std::atomic<int> g_sched_bwd_pair{-1};
constexpr int kHostChunks = 8;  // most head chunks of fa_fwd_host (events kept per device)

// Whether a forward call with a workspace can run the split schedule (D = 64 halves); use_split
// below decides whether it does.
bool split_capable(int D, int dtype) { return D == 64 && dtype != FA_F32; }

// Units of the D=64 forward's split schedule: the key blocks of each query-tile pair's tile 0
// (causal: min(nkb, 2p + 1) for pair p of a head, so p^2 of them before pair p while
// 2p - 1 < nkb, nkb per pair after that).
long long split_units(int BH, int M, int N, int causal) {
  const long long pairs = (M + 255) / 256, nkb = (N + 127) / 128;
  long long per_head = pairs * nkb;
  if (causal) {
    const long long c = (nkb + 1) / 2;
    per_head = pairs <= c ? pairs * pairs : c * c + (pairs - c) * nkb;
  }
  return static_cast<long long>(BH) * per_head;
}

// Whether the D = 64 forward takes the split schedule (fa_fwd_ws). Estimated times in key blocks
// per SM: whole pairs take rounds * nkb; the split takes its share, units / num_sms, plus about
// 3.5 blocks for its piece boundaries and merge, plus 1.2 for each further partial the holder of
// a pair's first blocks merges (a pair spans about nkb / share shares). Fitted to back-to-back
// times at fourteen non-causal shapes from B1 H2 N1024 to B16 H16 N4096 (a block is about
// 1.27 us): the split wins when pairs have many key blocks and either fill fewer SMs than there
// are or leave the last round part-empty (B1 H1 N8192 31.6 against 80.5 us, B1 H4 N2048 18.8
// against 24.3, B4 H12 N2048 60.5 against 65.1); whole pairs win with few key blocks a pair
// (B2 H12 N1024 15.4 against 18.1 us, B4 H12 N512 even). Within 3 % the call keeps whole pairs,
// whose schedule has no waits between CTAs.
bool use_split(int BH, int M, int N, int causal, int num_sms) {
  const long long pairs = static_cast<long long>(BH) * ((M + 255) / 256);
  const long long units = split_units(BH, M, N, causal);
  if (units >= (1ll << 31)) return false;  // the kernel indexes units in 32 bits
  const int forced = g_sched_fwd_split.load();
  if (forced >= 0) return forced == 1;
  const double nkb = static_cast<double>((N + 127) / 128);
  const double share = static_cast<double>(units) / num_sms;
  const double partials = std::max(0.0, std::ceil(nkb / share) - 1.0);
  const double split = share + 3.5 + 1.2 * partials;
  if (causal) {
    // whole pairs dealt in a serpentine order (heaviest with lightest) measured faster than the
    // split from a round of pairs up (B4 H12 N2048 44.1 against 50.9 us, B1 H16 N8192 151 against
    // 167): the split's extra pieces cost more than the balance gains. With fewer pairs than SMs
    // each pair has an SM and the call takes as long as the heaviest, tile 0 of a head's last pair
    // (B1 H4 N4096: 44.0 us whole, 25.4 split; B4 H12 N512 and N1024 stay whole).
    if (pairs >= num_sms) return false;
    const double pph = static_cast<double>((M + 255) / 256);
    return split < 0.97 * std::min(nkb, 2.0 * pph - 1.0);
  }
  const double rounds = static_cast<double>((pairs + num_sms - 1) / num_sms);
  return split < 0.97 * rounds * nkb;
}

// Whether the fused backward (fa_bwd_ws, D = 64) runs its split schedule (non-causal calls only).
// Estimated times in (key tile, query block) steps per SM: whole key tiles take rounds * nqb;
// the split takes its share, units / num_sms, plus about 5 steps for its piece boundaries and
// merge, plus 0.8 for each further partial the holder of a key tile's first blocks adds (a tile
// spans about nqb / share shares). Fitted to back-to-back times at twelve shapes (a step is
// 1.2-1.9 us): the split wins where key tiles have many query blocks and fill few SMs or leave
// the last round part-empty (B1 H1 N4096 34.3 against 58.9 us, B4 H12 N2048 163.4 against 180.3,
// B1 H4 N2048 31.8 against 35.8); whole tiles win with few query blocks a tile or many tiles
// (B1 H16 N1024 25.2 against 31.4 us, B4 H12 N1024 59.0 against 61.5, B8 H16 N2048 418 against
// 454). Within 3 % the call keeps whole tiles. fa_set_schedule(FA_SCHED_BWD_SPLIT, 0 / 1) forces
// it off / on (non-causal only).
bool use_bwd_split(int BH, int M, int N, int D, int causal, int num_sms) {
  if (D != 64 || causal) return false;
  const long long items = static_cast<long long>(BH) * ((N + 127) / 128);
  const long long nqb = (M + 127) / 128;
  const long long units = items * nqb;
  if (units >= (1ll << 31)) return false;  // the kernel indexes units in 32 bits
  const int forced = g_sched_bwd_split.load();
  if (forced >= 0) return forced == 1;
  const double share = static_cast<double>(units) / num_sms;
  const double partials = std::max(0.0, std::ceil(static_cast<double>(nqb) / share) - 1.0);
  const double rounds = static_cast<double>((items + num_sms - 1) / num_sms);
  return share + 5.0 + 0.8 * partials < 0.97 * rounds * static_cast<double>(nqb);
}

// Launch epochs of the split schedules' flags and counters. The sequence starts at a value
// drawn from the clock, so a word that foreign data left in a reused workspace is unlikely to
// equal the epoch of any launch; 0 (what a zero-filled workspace holds) is skipped.
uint32_t next_epoch() {
  static std::atomic<uint32_t> epoch{[] {
    uint64_t x = static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) +
                 0x9E3779B97F4A7C15ull;  // splitmix64 finaliser over the clock
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return static_cast<uint32_t>(x ^ (x >> 31));
  }()};
  uint32_t e = epoch.fetch_add(1u) + 1u;
  if (e == 0u) e = epoch.fetch_add(1u) + 1u;
  return e;
}
std::atomic<int> g_inject{0};  // fa_debug_inject: consumed by the next launch of the kind it names

// The pending injection if it is one of `a` or `b` (and then it is consumed), else 0.
int take_inject(int a, int b) {
  int k = g_inject.load();
  while ((k == a || k == b) && k != 0) {
    if (g_inject.compare_exchange_weak(k, 0)) return k;
  }
  return 0;
}

// fa_decode / fa_decode_ex: R query rows per (batch, head), each against all N keys.
fa_status decode_impl(const void* q, const void* Kcache, const void* Vcache, void* O, float* LSE, float* partial_ws,
                      int B, int H, int R, int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream,
                      const char* name) {
  FA_TRY(check_dtype(dtype));
  FA_TRY(check_sizes(B, H, 1, N, D));
  FA_TRY(check_scale(scale));
  if (R < 1) return fail(FA_ERR_INVALID, "%s: R=%d query rows", name, R);
  if (R > kDecMaxRows)
    return fail(FA_ERR_UNSUPPORTED, "%s: R=%d query rows above %d (fa_fwd takes any number)", name, R, kDecMaxRows);
  if (B * H == 0) return FA_OK;
  if (N == 0) return fail(FA_ERR_INVALID, "N = 0: softmax over an empty key set");
  if (n_splits < 1 || n_splits > N || n_splits > 65535)
    return fail(FA_ERR_INVALID, "n_splits=%d outside [1, min(N=%d, 65535)]", n_splits, N);
  if (B * H > 65535) return fail(FA_ERR_UNSUPPORTED, "%s: B*H=%d above 65535", name, B * H);
  FA_TRY(check_ptr(q, "q"));
  FA_TRY(check_ptr(Kcache, "Kcache"));
  FA_TRY(check_ptr(Vcache, "Vcache"));
  FA_TRY(check_ptr(O, "O"));
  FA_TRY(check_ptr(partial_ws, "partial_ws"));
  if (LSE != nullptr) FA_TRY(check_ptr(LSE, "LSE"));
  LaunchCtx ctx{};
  FA_TRY(make_ctx(&ctx, stream));
  ctx.inject = take_inject(kInjectDecodeStage, 0);
  cudaError_t e = launch_decode(q, Kcache, Vcache, O, LSE, partial_ws, B * H, R, N, D, scale, n_splits, dtype, ctx);
  if (e == cudaErrorNotSupported) return fail(FA_ERR_UNSUPPORTED, "%s: configuration not supported", name);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return FA_OK;
}

fa_status fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, void* ws, size_t ws_bytes, int B,
                   int H, int M, int N, int D, float scale, int causal, fa_dtype dtype, void* stream,
                   const char* name) {
  FA_TRY(check_dtype(dtype));
  FA_TRY(check_sizes(B, H, M, N, D));
  FA_TRY(check_scale(scale));
  if (B * H == 0 || M == 0) return FA_OK;
  if (N == 0) return fail(FA_ERR_INVALID, "N = 0: softmax over an empty key set");
  FA_TRY(check_ptr(Q, "Q"));
  FA_TRY(check_ptr(K, "K"));
  FA_TRY(check_ptr(V, "V"));
  FA_TRY(check_ptr(O, "O"));
  if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return fail(FA_ERR_INVALID, "LSE misaligned");
  LaunchCtx ctx{};
  FA_TRY(make_ctx(&ctx, stream));
  if (D == 64 && dtype != FA_F32) ctx.inject = take_inject(kInjectFwdStage, kInjectFwdFlag);
  FwdSplit sp{};
  if (ws != nullptr && split_capable(D, dtype)) {
    FA_TRY(check_ptr(ws, "workspace"));
    const size_t need = fwd_d64_split_bytes(ctx.num_sms);
    if (ws_bytes < need) return fail(FA_ERR_INVALID, "%s: workspace of %zu bytes, %zu needed", name, ws_bytes, need);
    if (use_split(B * H, M, N, causal, ctx.num_sms)) {
      sp.ws = static_cast<float*>(ws);
      sp.flags = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + need - ctx.num_sms * 8 * sizeof(uint32_t));
      sp.epoch = next_epoch();
    }
  }
  int parts = 1;
  size_t split_bytes = 0;
  if (dtype == FA_F32 && ws != nullptr && D == 64) {
    parts = fwd_f32_parts(B * H, M, N, ctx.num_sms);
    split_bytes = align256(fwd_f32_split_bytes(B * H, M, parts));
    const size_t need = split_bytes + fwd_f32_presplit_bytes(B * H, N);
    FA_TRY(check_ptr(ws, "workspace"));
    if (ws_bytes < need) return fail(FA_ERR_INVALID, "%s: workspace of %zu bytes, %zu needed", name, ws_bytes, need);
  }
  cudaError_t e;
  if (dtype == FA_F32) {
    uint32_t ep = 0;
    if (parts > 1) ep = next_epoch();
    if (ws != nullptr && D == 64)  // operands split once by a prologue, pipelined main kernel
      e = launch_fwd_f32_presplit(Q, K, V, O, LSE, B * H, M, N, scale, causal != 0, parts, static_cast<float*>(ws),
                                  ep, static_cast<char*>(ws) + split_bytes, ctx);
    else
      e = launch_fwd_f32(Q, K, V, O, LSE, B * H, M, N, D, scale, causal != 0, 1, nullptr, 0, ctx);
  } else {
    e = launch_fwd_half(Q, K, V, O, LSE, B * H, M, N, D, scale, causal != 0, dtype, sp, ctx);
  }
  if (e == cudaErrorNotSupported) return fail(FA_ERR_UNSUPPORTED, "%s: configuration not supported", name);
  if (e == cudaErrorInvalidValue) return fail(FA_ERR_CUDA, "%s: TMA descriptor rejected by the driver", name);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return FA_OK;
}

// fa_bwd / fa_bwd_ws: delta_ws holds delta (B*H*M f32); dQacc, when not null, the fused path's f32
// dQ accumulator (B*H*M*64).
fa_status bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                   void* dQ, void* dK, void* dV, float* delta_ws, float* dQacc, float* split_ws, int B, int H, int M,
                   int N, int D, float scale, int causal, fa_dtype dtype, void* stream, const char* name) {
  FA_TRY(check_dtype(dtype));
  FA_TRY(check_sizes(B, H, M, N, D));
  if (dtype == FA_F32) return fail(FA_ERR_UNSUPPORTED, "%s supports FA_F16 and FA_BF16", name);
  FA_TRY(check_scale(scale));
  if (B * H == 0 || M == 0) return FA_OK;
  if (N == 0) return fail(FA_ERR_INVALID, "N = 0: softmax over an empty key set");
  FA_TRY(check_ptr(Q, "Q"));
  FA_TRY(check_ptr(K, "K"));
  FA_TRY(check_ptr(V, "V"));
  FA_TRY(check_ptr(O, "O"));
  FA_TRY(check_ptr(dO, "dO"));
  FA_TRY(check_ptr(LSE, "LSE"));
  FA_TRY(check_ptr(dQ, "dQ"));
  FA_TRY(check_ptr(dK, "dK"));
  FA_TRY(check_ptr(dV, "dV"));
  FA_TRY(check_ptr(delta_ws, "delta_ws"));
  LaunchCtx ctx{};
  FA_TRY(make_ctx(&ctx, stream));
  BwdSplit sp{};
  if (dQacc != nullptr && split_ws != nullptr && use_bwd_split(B * H, M, N, D, causal, ctx.num_sms)) {
    sp.ws = split_ws;
    ctx.inject = take_inject(kInjectBwdCount, 0);
  }
  // fa_bwd's dK/dV and dQ kernels at D = 64 on CTA pairs: by default only for non-causal calls
  // with fewer key tiles than SMs, where they measured 4-7 % faster (Z1 H2 N1024: 30.7 against
  // 32.8 us). With a wave or more of key tiles the single-CTA kernels are 2-3 % faster (B4 H12
  // N2048: 251 against 257 us); causal calls keep single CTAs (a pair's 256 rows walk the blocks
  // of its later half, so the earlier CTA gets one wholly masked block per item, and the items are
  // coarser to balance).
  const int pair_forced = g_sched_bwd_pair.load();
  const long long key_tiles = static_cast<long long>(B) * H * ((N + 127) / 128);
  sp.pair = dQacc == nullptr && D == 64 &&
            (pair_forced == 1 || (pair_forced == -1 && causal == 0 && key_tiles < ctx.num_sms));
  cudaError_t e =
      launch_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, delta_ws, dQacc, B * H, M, N, D, scale, causal != 0, dtype, sp, ctx);
  if (e == cudaErrorNotSupported) return fail(FA_ERR_UNSUPPORTED, "%s: configuration not supported", name);
  if (e == cudaErrorInvalidValue) return fail(FA_ERR_CUDA, "%s: TMA descriptor rejected by the driver", name);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return FA_OK;
}

}  // namespace

namespace fa {
fa_status decode_entry(const void* q, const void* Kcache, const void* Vcache, void* O, float* LSE, float* partial_ws,
                       int B, int H, int R, int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream,
                       const char* name) {
  return decode_impl(q, Kcache, Vcache, O, LSE, partial_ws, B, H, R, N, D, scale, n_splits, dtype, stream, name);
}
fa_status fail_msg(fa_status s, const char* msg) { return fail(s, "%s", msg); }
fa_status cuda_fail_msg(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace fa

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID: return "FA_ERR_INVALID: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported configuration";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA error";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "unknown fa_status";
}

const char* fa_last_error_message(void) { return t_msg; }

fa_status fa_set_wait_budget_ns(unsigned long long ns) {
  if (ns < 1000ull) return fail(FA_ERR_INVALID, "wait budget %llu ns is below 1000 ns", ns);
  std::lock_guard<std::mutex> lock(g_mutex);
  g_wait_budget_ns = ns;
  return FA_OK;
}

fa_status fa_set_schedule(fa_sched_key key, int value) {
  switch (key) {
    case FA_SCHED_FWD_SPLIT:
    case FA_SCHED_BWD_SPLIT:
      if (value < -1 || value > 1) return fail(FA_ERR_INVALID, "schedule key %d takes -1, 0 or 1 (got %d)", key, value);
      (key == FA_SCHED_FWD_SPLIT ? g_sched_fwd_split : g_sched_bwd_split).store(value);
      return FA_OK;
    case FA_SCHED_BWD_PAIR:
      if (value < -1 || value > 1) return fail(FA_ERR_INVALID, "schedule key %d takes -1, 0 or 1 (got %d)", key, value);
      g_sched_bwd_pair.store(value);
      return FA_OK;
    case FA_SCHED_HOST_CHUNKS:
      if (value != -1 && (value < 1 || value > kHostChunks))
        return fail(FA_ERR_INVALID, "host chunks take -1 or 1..%d (got %d)", kHostChunks, value);
      g_sched_host_chunks.store(value);
      return FA_OK;
  }
  return fail(FA_ERR_INVALID, "unknown schedule key %d", static_cast<int>(key));
}

fa_status fa_debug_inject(int kind) {
  if (kind < 0 || kind > kInjectBwdCount) return fail(FA_ERR_INVALID, "unknown fault-injection kind %d", kind);
  g_inject.store(kind);
  return FA_OK;
}

int fa_debug_schedule_choice(int which, int B, int H, int M, int N, int causal, int num_sms) {
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0 || num_sms <= 0) return -1;
  if (static_cast<long long>(B) * H > INT_MAX) return -1;
  if (which == 0) return use_split(B * H, M, N, causal, num_sms) ? 1 : 0;
  if (which == 1) return use_bwd_split(B * H, M, N, 64, causal, num_sms) ? 1 : 0;
  return -1;
}

size_t fa_bwd_workspace_bytes(int B, int H, int M) {
  if (B <= 0 || H <= 0 || M <= 0) return 0;
  return static_cast<size_t>(B) * H * M * sizeof(float);
}

size_t fa_decode_workspace_bytes(int B, int H, int D, int n_splits) {
  if (B <= 0 || H <= 0 || D <= 0 || n_splits <= 0) return 0;
  return static_cast<size_t>(B) * H * n_splits * (D + 2) * sizeof(float);
}

size_t fa_decode_ex_workspace_bytes(int B, int H, int R, int D, int n_splits) {
  if (B <= 0 || H <= 0 || R <= 0 || D <= 0 || n_splits <= 0) return 0;
  return static_cast<size_t>(B) * H * R * n_splits * (D + 2) * sizeof(float);
}

size_t fa_fwd_workspace_bytes(int B, int H, int M, int N, int D, int causal, fa_dtype dtype) {
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0) return 0;
  DevState* st = nullptr;
  if (device_state(&st) != FA_OK) return 0;
  if (dtype == FA_F32 && D == 64)  // the split's partials, then K and V split into tf32 parts
    return align256(fwd_f32_split_bytes(B * H, M, fwd_f32_parts(B * H, M, N, st->num_sms))) +
           fwd_f32_presplit_bytes(B * H, N);
  if (!split_capable(D, dtype)) return 0;
  return fwd_d64_split_bytes(st->num_sms);
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int M, int N, int D,
                 float scale, int causal, fa_dtype dtype, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, nullptr, 0, B, H, M, N, D, scale, causal, dtype, stream, "fa_fwd");
}

fa_status fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE, void* workspace,
                    size_t workspace_bytes, int B, int H, int M, int N, int D, float scale, int causal, fa_dtype dtype,
                    void* stream) {
  return fwd_impl(Q, K, V, O, LSE, workspace, workspace_bytes, B, H, M, N, D, scale, causal, dtype, stream,
                  "fa_fwd_ws");
}


fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                 void* dQ, void* dK, void* dV, float* delta_ws, int B, int H, int M, int N, int D, float scale,
                 int causal, fa_dtype dtype, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, delta_ws, nullptr, nullptr, B, H, M, N, D, scale, causal, dtype,
                  stream, "fa_bwd");
}

// workspace of fa_bwd_ws: delta, then (D = 64) the f32 dQ accumulator and the split schedule's
// partial slots and flags, each 256-byte aligned
size_t fa_bwd_ws_workspace_bytes(int B, int H, int M, int D) {
  if (B <= 0 || H <= 0 || M <= 0 || D <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H * M;
  const size_t delta = (rows * sizeof(float) + 255u) & ~static_cast<size_t>(255u);
  if (D != 64) return delta;
  DevState* st = nullptr;
  if (device_state(&st) != FA_OK) return 0;
  return delta + rows * 64 * sizeof(float) + bwd_fused_split_bytes(st->num_sms);
}

fa_status fa_bwd_ws(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                    void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int M, int N,
                    int D, float scale, int causal, fa_dtype dtype, void* stream) {
  const size_t need = fa_bwd_ws_workspace_bytes(B, H, M, D);
  if (B * H > 0 && M > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(FA_ERR_INVALID, "fa_bwd_ws: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  float* delta = static_cast<float*>(workspace);
  float* acc = nullptr;
  float* split = nullptr;
  if (D == 64 && B * H > 0 && M > 0) {
    const size_t rows = static_cast<size_t>(B) * H * M;
    acc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                   ((rows * sizeof(float) + 255u) & ~static_cast<size_t>(255u)));
    split = acc + rows * 64;  // rows * 256 bytes past a 256-byte boundary
  }
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, delta, acc, split, B, H, M, N, D, scale, causal, dtype, stream,
                  "fa_bwd_ws");
}

fa_status fa_decode(const void* q, const void* Kcache, const void* Vcache, void* O, float* partial_ws, int B, int H,
                    int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream) {
  return decode_impl(q, Kcache, Vcache, O, nullptr, partial_ws, B, H, 1, N, D, scale, n_splits, dtype, stream,
                     "fa_decode");
}

fa_status fa_decode_ex(const void* q, const void* Kcache, const void* Vcache, void* O, float* LSE, float* partial_ws,
                       int B, int H, int R, int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream) {
  return decode_impl(q, Kcache, Vcache, O, LSE, partial_ws, B, H, R, N, D, scale, n_splits, dtype, stream,
                     "fa_decode_ex");
}

// ---------------------------------------------------------------------------
// FP8 forward: the workspace holds the E4M3 operands and their scales (see Fp8Ws).
namespace {
struct Fp8Layout {
  size_t q8, k8, vt8, sq, sk, vmax, sv, total;
  int npad;
};
Fp8Layout fp8_layout(int B, int H, int M, int N) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t nqb = (static_cast<size_t>(M) + 127) / 128, nkb = (static_cast<size_t>(N) + 127) / 128;
  auto a256 = [](size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); };
  Fp8Layout L{};
  L.npad = (N + 15) / 16 * 16;
  L.q8 = 0;
  L.k8 = L.q8 + a256(BH * M * 64);
  L.vt8 = L.k8 + a256(BH * N * 64);
  L.sq = L.vt8 + a256(BH * 64 * static_cast<size_t>(L.npad));
  L.sk = L.sq + a256(BH * nqb * 4);
  L.vmax = L.sk + a256(BH * nkb * 4);
  L.sv = L.vmax + a256(BH * nkb * 4);
  L.total = L.sv + a256(BH * 4);
  return L;
}
}  // namespace

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int M, int N, int D) {
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0 || D != 64) return 0;
  return fp8_layout(B, H, M, N).total;
}

fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE, const signed char* signs,
                     void* workspace, size_t workspace_bytes, int B, int H, int M, int N, int D, float scale,
                     int causal, fa_dtype dtype, void* stream) {
  FA_TRY(check_dtype(dtype));
  FA_TRY(check_sizes(B, H, M, N, D));
  if (dtype == FA_F32) return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8: inputs must be FA_F16 or FA_BF16");
  if (D != 64) return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8: head dimension D=%d (supported: 64)", D);
  FA_TRY(check_scale(scale));
  if (B * H == 0 || M == 0) return FA_OK;
  if (N == 0) return fail(FA_ERR_INVALID, "N = 0: softmax over an empty key set");
  if (B * H > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8: B*H=%d above 65535", B * H);
  FA_TRY(check_ptr(Q, "Q"));
  FA_TRY(check_ptr(K, "K"));
  FA_TRY(check_ptr(V, "V"));
  FA_TRY(check_ptr(O, "O"));
  FA_TRY(check_ptr(signs, "signs"));  // read 16 bytes at a time
  if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return fail(FA_ERR_INVALID, "LSE misaligned");
  FA_TRY(check_ptr(workspace, "workspace"));
  const Fp8Layout L = fp8_layout(B, H, M, N);
  if (workspace_bytes < L.total)
    return fail(FA_ERR_INVALID, "fa_fwd_fp8: workspace of %zu bytes, %zu needed", workspace_bytes, L.total);
  LaunchCtx ctx{};
  FA_TRY(make_ctx(&ctx, stream));
  char* ws = static_cast<char*>(workspace);
  Fp8Ws w{};
  w.q8 = reinterpret_cast<uint8_t*>(ws + L.q8);
  w.k8 = reinterpret_cast<uint8_t*>(ws + L.k8);
  w.vt8 = reinterpret_cast<uint8_t*>(ws + L.vt8);
  w.sq = reinterpret_cast<float*>(ws + L.sq);
  w.sk = reinterpret_cast<float*>(ws + L.sk);
  w.vmax = reinterpret_cast<float*>(ws + L.vmax);
  w.sv = reinterpret_cast<float*>(ws + L.sv);
  w.npad = L.npad;
  cudaError_t e = launch_fp8_quant(Q, K, V, reinterpret_cast<const int8_t*>(signs), w, B * H, M, N, dtype, ctx.stream);
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_fp8: quantisation launch");
  e = launch_fwd_fp8(w, O, LSE, B * H, M, N, scale, causal != 0, dtype, ctx);
  if (e == cudaErrorInvalidValue) return fail(FA_ERR_CUDA, "fa_fwd_fp8: TMA descriptor rejected by the driver");
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_fp8");
  return FA_OK;
}

fa_status fa_last_status(void* stream) {
  DevState* st = nullptr;
  FA_TRY(device_state(&st));
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DevStatus h{};
  e = cudaMemcpy(&h, st->status, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (h.code == 0u) return FA_OK;
  DevStatus zero{};
  e = cudaMemcpy(st->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  static const char* names[] = {"?", "fwd", "fwd_f32", "bwd_delta", "bwd_dkdv", "bwd_dq", "decode_split",
                                "decode_combine", "fwd_fp8"};
  const char* kn = h.kernel < 9 ? names[h.kernel] : "?";
  if (h.code == kStatusTimeout)
    return fail(FA_ERR_TIMEOUT, "kernel %s gave up wait site %u in block %u", kn, h.site, h.block);
  return fail(FA_ERR_CUDA, "kernel %s reported status %u (site %u, block %u)", kn, h.code, h.site, h.block);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward on host buffers, with the copies overlapped with the kernels.
//
// The (batch, head) heads are cut into chunks: by default three, of about 4/7, 2/7 and 1/7 of
// the heads (fa_set_schedule with FA_SCHED_HOST_CHUNKS fixes a count of equal chunks instead,
// 1..8). Three internal streams of the device carry the copies in, the kernels and the copies
// out, so chunk c's inputs travel while chunk c-1 is computed and earlier chunks' outputs travel
// back; events order each chunk's three steps, and the caller's stream is joined at entry and at
// exit, so the call is ordered on it like any other.

namespace {

// The copies in and out share the host link (about 245 GB/s together, 200 one way), and a
// chunk's outputs can only leave after its kernel: the time after the last input lands is that
// chunk's kernel and its copy out, so the last chunk is the smallest. At B4 H12 N2048 D64 (a
// per-chunk event timeline) chunks of 28, 14 and 6 heads took 281-285 us a call against 298-307
// for three equal chunks and 306-315 for four; more chunks add per-copy and per-launch costs.
constexpr int kHostDefaultChunks = 3;

// First head of chunk c of n over BH heads (c = n gives BH).
long long host_chunk_start(long long BH, int n, int c, bool equal) {
  if (equal || n != kHostDefaultChunks) return static_cast<long long>(c) * BH / n;
  static const int kSevenths[kHostDefaultChunks + 1] = {0, 4, 6, 7};  // 4:2:1
  return (BH * kSevenths[c] + 3) / 7;
}

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, finish = nullptr;
  cudaEvent_t in[kHostChunks] = {}, done[kHostChunks] = {};
};

HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;  // the internal streams are shared by every caller of a device

fa_status host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_CUDA, "device ordinal %d out of range", dev);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    for (cudaStream_t* s : {&hp.h2d, &hp.comp, &hp.d2h}) {
      e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
      if (e != cudaSuccess) return cuda_fail(e, "creating the copy/compute streams");
    }
    std::vector<cudaEvent_t*> evs = {&hp.start, &hp.finish};
    for (int c = 0; c < kHostChunks; ++c) {
      evs.push_back(&hp.in[c]);
      evs.push_back(&hp.done[c]);
    }
    for (cudaEvent_t* ev : evs) {
      e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(e, "creating the pipeline events");
    }
    hp.ready = true;
  }
  *out = &hp;
  return FA_OK;
}

// Device workspace of fa_fwd_host: the forward's own workspace for the largest chunk, then
// Q, K, V, O and LSE of the whole problem, each 256-byte aligned.
struct HostLayout {
  int chunks = 0;
  bool equal = true;  // equal chunks, or the default 4:2:1 cut
  size_t split = 0, q = 0, k = 0, v = 0, o = 0, lse = 0, total = 0;
};

HostLayout host_layout(int B, int H, int M, int N, int D, int causal, fa_dtype dtype) {
  HostLayout L;
  const long long BH = static_cast<long long>(B) * H;
  const int forced = g_sched_host_chunks.load();
  const int want = forced >= 1 ? forced : kHostDefaultChunks;
  L.chunks = static_cast<int>(BH < want ? BH : want);
  L.equal = forced >= 1 || BH < 7;  // the 4:2:1 cut needs a head in its smallest chunk
  size_t w = 0;  // the forward's own workspace, for the largest chunk
  for (int c = 0; c < L.chunks; ++c) {
    const long long nh = host_chunk_start(BH, L.chunks, c + 1, L.equal) - host_chunk_start(BH, L.chunks, c, L.equal);
    const size_t wc = nh > 0 ? fa_fwd_workspace_bytes(1, static_cast<int>(nh), M, N, D, causal, dtype) : 0;
    w = wc > w ? wc : w;
  }
  const size_t es = dtype == FA_F32 ? 4 : 2;
  const size_t qb = static_cast<size_t>(BH) * M * D * es, kb = static_cast<size_t>(BH) * N * D * es;
  L.split = 0;
  L.q = align256(w);
  L.k = L.q + align256(qb);
  L.v = L.k + align256(kb);
  L.o = L.v + align256(kb);
  L.lse = L.o + align256(qb);
  L.total = L.lse + align256(static_cast<size_t>(BH) * M * sizeof(float));
  return L;
}

}  // namespace

extern "C" {

size_t fa_fwd_host_workspace_bytes(int B, int H, int M, int N, int D, int causal, fa_dtype dtype) {
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0 || D <= 0) return 0;
  if (check_dtype(dtype) != FA_OK) return 0;
  return host_layout(B, H, M, N, D, causal, dtype).total;
}

fa_status fa_fwd_host(const void* hQ, const void* hK, const void* hV, void* hO, float* hLSE, void* dev_ws,
                      size_t dev_ws_bytes, int B, int H, int M, int N, int D, float scale, int causal, fa_dtype dtype,
                      void* stream) {
  FA_TRY(check_dtype(dtype));
  FA_TRY(check_sizes(B, H, M, N, D));
  FA_TRY(check_scale(scale));
  if (B * H == 0 || M == 0) return FA_OK;
  if (N == 0) return fail(FA_ERR_INVALID, "N = 0: softmax over an empty key set");
  // what the forward supports, checked before anything is queued
  if ((D != 64 && D != 128) || (dtype == FA_F32 && D != 64))
    return fail(FA_ERR_UNSUPPORTED, "fa_fwd_host: D=%d not supported for this dtype", D);
  if (hQ == nullptr || hK == nullptr || hV == nullptr || hO == nullptr)
    return fail(FA_ERR_INVALID, "fa_fwd_host: a host buffer is NULL");
  FA_TRY(check_ptr(dev_ws, "dev_ws"));
  const HostLayout L = host_layout(B, H, M, N, D, causal, dtype);
  if (dev_ws_bytes < L.total)
    return fail(FA_ERR_INVALID, "fa_fwd_host: dev_ws of %zu bytes, %zu needed", dev_ws_bytes, L.total);
  HostPipe* hp = nullptr;
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  FA_TRY(host_pipe(&hp));
  char* ws = static_cast<char*>(dev_ws);
  const size_t es = dtype == FA_F32 ? 4 : 2;
  const size_t qrow = static_cast<size_t>(M) * D * es, krow = static_cast<size_t>(N) * D * es;  // per head
  const int BH = B * H;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaEventRecord(hp->start, user);
  for (cudaStream_t s : {hp->h2d, hp->comp, hp->d2h})
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_host: joining the caller's stream");
  for (int c = 0; c < L.chunks; ++c) {
    const int h0 = static_cast<int>(host_chunk_start(BH, L.chunks, c, L.equal));
    const int h1 = static_cast<int>(host_chunk_start(BH, L.chunks, c + 1, L.equal));
    const int nh = h1 - h0;
    char* dq = ws + L.q + h0 * qrow;
    char* dk = ws + L.k + h0 * krow;
    char* dv = ws + L.v + h0 * krow;
    char* dout = ws + L.o + h0 * qrow;
    float* dl = reinterpret_cast<float*>(ws + L.lse) + static_cast<size_t>(h0) * M;
    e = cudaMemcpyAsync(dq, static_cast<const char*>(hQ) + h0 * qrow, nh * qrow, cudaMemcpyHostToDevice, hp->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dk, static_cast<const char*>(hK) + h0 * krow, nh * krow, cudaMemcpyHostToDevice, hp->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dv, static_cast<const char*>(hV) + h0 * krow, nh * krow, cudaMemcpyHostToDevice, hp->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(hp->in[c], hp->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->in[c], 0);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_host: copy in");
    const fa_status s = fwd_impl(dq, dk, dv, dout, hLSE != nullptr ? dl : nullptr, ws + L.split, L.q, 1, nh, M, N, D,
                                 scale, causal, dtype, hp->comp, "fa_fwd_host");
    if (s != FA_OK) return s;
    e = cudaEventRecord(hp->done[c], hp->comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->done[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(hO) + h0 * qrow, dout, nh * qrow, cudaMemcpyDeviceToHost, hp->d2h);
    if (e == cudaSuccess && hLSE != nullptr)
      e = cudaMemcpyAsync(hLSE + static_cast<size_t>(h0) * M, dl, static_cast<size_t>(nh) * M * sizeof(float),
                          cudaMemcpyDeviceToHost, hp->d2h);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_host: copy out");
  }
  e = cudaEventRecord(hp->finish, hp->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(user, hp->finish, 0);
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_host: joining the caller's stream");
  return FA_OK;
}

}  // extern "C"
