// ssm_abi.cu -- the extern "C" boundary of libssm_b300.so (declared in include/ssm.h).
//
// Host side only: validate every descriptor, pick a kernel variant, enqueue it on the
// caller's stream. Nothing here allocates, frees or synchronises (except the explicit
// diagnostic ssm_device_error).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <initializer_list>
#include <mutex>

#include "../../include/ssm.h"
#include "common.cuh"
#include "scan_fwd.cuh"
#include "scan_bwd.cuh"
#include "scan_fwd_chan.cuh"
#include "ssd_fwd.cuh"
#include "state_update.cuh"
#include "state_update_stream.cuh"

namespace {

using ssm::DecodeParams;
using ssm::FwdParams;

bool dtype_ok(ssm_dtype_t t) { return t == SSM_F32 || t == SSM_BF16; }
int64_t elem_size(ssm_dtype_t t) { return t == SSM_F32 ? 4 : 2; }

int64_t numel(const ssm_tensor_t* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// Shape, non-null data and alignment of one descriptor: natural element alignment
// always, 16 bytes where a kernel reads the tensor with 16-byte vectors (align16).
ssm_status_t check_tensor(const ssm_tensor_t* t, std::initializer_list<int64_t> shape, bool align16 = false) {
  if (!t) return SSM_ERR_NULL;
  if (t->ndim != (int32_t)shape.size() || t->ndim < 1 || t->ndim > 3) return SSM_ERR_SHAPE;
  int i = 0;
  for (int64_t s : shape) {
    if (t->shape[i] != s || s < 0) return SSM_ERR_SHAPE;
    ++i;
  }
  if (!dtype_ok(t->dtype)) return SSM_ERR_DTYPE;
  if (numel(t) > 0) {
    if (!t->data) return SSM_ERR_NULL;
    const uintptr_t a = reinterpret_cast<uintptr_t>(t->data);
    if (a % (uintptr_t)elem_size(t->dtype) != 0 || (align16 && a % 16 != 0)) return SSM_ERR_LAYOUT;
  }
  return SSM_OK;
}

struct Span {
  uintptr_t lo = 0, hi = 0;  // [lo, hi)
};
Span span_of(const ssm_tensor_t* t) {
  Span s;
  if (t && t->data && numel(t) > 0) {
    s.lo = reinterpret_cast<uintptr_t>(t->data);
    s.hi = s.lo + (uintptr_t)(numel(t) * elem_size(t->dtype));
  }
  return s;
}
bool overlaps(const ssm_tensor_t* a, const ssm_tensor_t* b) {
  Span x = span_of(a), y = span_of(b);
  if (x.lo == x.hi || y.lo == y.hi) return false;
  return x.lo < y.hi && y.lo < x.hi;
}

bool n_supported(int64_t n) { return n == 4 || n == 8 || n == 16; }

// ---- kernel-variant selection ------------------------------------------------------
// SSM_B300_FORWARD_KERNEL = auto (default) | generic | chan. Both variants compute the
// same result; the override exists so each can be checked on its own.
enum class FwdVariant { kAuto, kGeneric, kChan };
FwdVariant forward_variant() {
  const char* e = getenv("SSM_B300_FORWARD_KERNEL");
  if (e && strcmp(e, "generic") == 0) return FwdVariant::kGeneric;
  if (e && strcmp(e, "chan") == 0) return FwdVariant::kChan;
  return FwdVariant::kAuto;
}

// ---- failure detection ---------------------------------------------------------------
// SSM_B300_WAIT_LIMIT_CYCLES: limit of the channel kernel's bounded waits (default about
// one second). SSM_B300_FAULT_INJECT=skip_loads: the channel kernel's TMA issuer issues
// nothing, so every wait for data runs out; only the failure-detection tests set it.
long long wait_limit_cycles() {
  const char* e = getenv("SSM_B300_WAIT_LIMIT_CYCLES");
  if (!e) return 0;
  const long long v = atoll(e);
  return v > 0 ? v : 0;
}
int fault_skip_loads() {
  const char* e = getenv("SSM_B300_FAULT_INJECT");
  return (e && strcmp(e, "skip_loads") == 0) ? 1 : 0;
}

// ---- TMA descriptors -------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Dense (batch, L, inner) tensor as a 3-D TMA map with box (1, box_l, box_inner); loads
// zero-fill and stores clip outside the tensor, so a chunk never crosses into the next
// batch row.
bool encode_3d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, uint64_t esize, uint64_t inner,
               uint64_t L, uint64_t batch, uint32_t box_inner, uint32_t box_l) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, L, batch};
  cuuint64_t strides[2] = {inner * esize, inner * L * esize};
  cuuint32_t box[3] = {box_inner, box_l, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// ---- channel-parallel TMA kernel (bf16 I/O) ----------------------------------------------
constexpr int kChanTC = 32, kChanStages = 4;

bool chan_eligible(const FwdParams& p, int64_t N) {
  // TMA needs 16-byte aligned bases and row pitches (D % 8 == 0 covers bf16 and fp32
  // y) and int32 coordinates; last_state is written with 16-byte vector stores.
  // The zero-order-hold B-bar runs here too, except with the conv prologue.
  return !(p.zoh && p.conv_w) && (N == 8 || N == 16) && p.D % 8 == 0 && p.L < (int64_t)INT32_MAX && aligned16(p.u) &&
         aligned16(p.delta) && aligned16(p.z) && aligned16(p.B) && aligned16(p.C) && aligned16(p.y) &&
         aligned16(p.last_state) && encode_fn() != nullptr;
}

template <typename TY, int N, bool kSP, bool kZ, bool kAgg, bool kConv, bool kCk = false, bool kZoh = false>
cudaError_t launch_chan_k(const FwdParams& p, const CUtensorMap* maps, int nseg, cudaStream_t st) {
  auto kern = &ssm::scan_fwd_chan<TY, N, kChanTC, kChanStages, kSP, kZ, kAgg, kConv, kCk, kZoh>;
  constexpr int smem = ssm::chan_smem_bytes<TY, N, kChanTC, kChanStages>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  dim3 grid((unsigned)((p.D + ssm::kChanCTA - 1) / ssm::kChanCTA), (unsigned)p.batch, (unsigned)nseg);
  void* args[] = {const_cast<CUtensorMap*>(&maps[0]), const_cast<CUtensorMap*>(&maps[1]),
                  const_cast<CUtensorMap*>(&maps[2]), const_cast<CUtensorMap*>(&maps[3]),
                  const_cast<CUtensorMap*>(&maps[4]), const_cast<CUtensorMap*>(&maps[5]),
                  const_cast<FwdParams*>(&p)};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), grid, dim3(ssm::kChanThreads), args, smem, st);
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// Segment length for nseg segments of a sequence of L steps: a multiple of the chunk tc,
// at least min_len, and with a last segment of at least `rows` steps (the segments keep
// their carries in their own first rows of y). Lowers nseg until that holds; returns the
// number of segments (< 2: do not segment) and the length in *len.
// SSM_B300_SEGMENTS=0 turns segmentation off: every pass then runs each recurrence in
// order from its start state, so splitting a sequence into a prefix and its continuation
// reproduces one pass bit for bit (segments reassociate the recurrence: equal up to
// rounding).
bool segments_enabled() {
  const char* e = getenv("SSM_B300_SEGMENTS");
  return !(e && strcmp(e, "0") == 0);
}

// SSM_B300_DECODE=plain: the decode step always uses the one-launch-per-thread kernel
// (tests compare it with the streamed one).
bool decode_streamed() {
  const char* e = getenv("SSM_B300_DECODE");
  return !(e && strcmp(e, "plain") == 0);
}

int64_t fit_segments(int64_t L, int64_t nseg, int64_t tc, int64_t min_len, int64_t rows, int64_t* len) {
  if (!segments_enabled()) return 1;
  for (; nseg >= 2; --nseg) {
    int64_t l = ((L + nseg - 1) / nseg + tc - 1) / tc * tc;
    if (l < min_len) l = min_len;
    const int64_t n = (L + l - 1) / l;
    if (n >= 2 && L - (n - 1) * l >= rows) {
      *len = l;
      return n;
    }
  }
  return 1;
}

// Sequence segmentation for shapes with too few channel blocks to occupy the GPU: the
// long sequence is cut into nseg segments of seg_len steps (a multiple of the chunk),
// each processed by its own CTAs; the workspace holds E, P and H ([nseg][batch][D][N]
// fp32 each).
struct SegPlan {
  int nseg = 1;
  int64_t seg_len = 0;
  size_t bytes = 0;
};
SegPlan plan_segments(int64_t batch, int64_t L, int64_t D, int64_t N) {
  SegPlan sp;
  sp.seg_len = L;
  const int sms = num_sms();
  const int64_t ctas = ((D + ssm::kChanCTA - 1) / ssm::kChanCTA) * batch;
  if (sms <= 0 || ctas <= 0 || ctas * 2 > sms) return sp;
  int64_t nseg = sms / ctas;
  if (nseg > 128) nseg = 128;  // the carry scan covers up to 4 warps x 32 segments
  if (nseg < 2) return sp;
  int64_t len = L;  // segments of at least 8 chunks: shorter ones do not pay for the aggregate pass
  nseg = fit_segments(L, nseg, kChanTC, 8 * kChanTC, 6 * N, &len);
  if (nseg < 2) return sp;
  sp.nseg = (int)nseg;
  sp.seg_len = len;
  sp.bytes = (size_t)3 * nseg * batch * D * N * sizeof(float);
  return sp;
}

// The carry scan over segments (block carry across warps above 32 segments): values in
// y (sy.y set) or in the flat workspace arrays E, P -> H.
cudaError_t launch_carry(const ssm::SegY& sy, const float* E, const float* P, const float* h0, float* H, int nseg,
                         int64_t nbdn, cudaStream_t st) {
  int wpi = (nseg + 31) / 32;
  if (wpi == 3) wpi = 4;
  const int64_t per_cta = 4 / wpi;
  void* args[] = {const_cast<ssm::SegY*>(&sy), &E, &P, &h0, &H, &nseg, &wpi, &nbdn};
  const void* kern = sy.y ? reinterpret_cast<const void*>(&ssm::seg_carry_kernel<true>)
                          : reinterpret_cast<const void*>(&ssm::seg_carry_kernel<false>);
  return cudaLaunchKernel(kern, dim3((unsigned)((nbdn + per_cta - 1) / per_cta)), dim3(128), args, 0, st);
}

// Run-time switches (softplus, gate, conv prologue) to template arguments. The
// aggregate pass never gates.
template <typename TY, int N, bool kAgg, bool kConv>
cudaError_t launch_chan_sz(const FwdParams& p, const CUtensorMap* maps, int nseg, cudaStream_t st, bool sp, bool z) {
  if (kAgg) z = false;
  if constexpr (!kConv) {
    if (p.zoh) {  // the zero-order-hold B-bar (not with checkpoints: the training pair is the Delta B form)
      if (sp && z) return launch_chan_k<TY, N, true, !kAgg, kAgg, false, false, true>(p, maps, nseg, st);
      if (sp) return launch_chan_k<TY, N, true, false, kAgg, false, false, true>(p, maps, nseg, st);
      if (z) return launch_chan_k<TY, N, false, !kAgg, kAgg, false, false, true>(p, maps, nseg, st);
      return launch_chan_k<TY, N, false, false, kAgg, false, false, true>(p, maps, nseg, st);
    }
  }
  if constexpr (!kAgg && !kConv) {
    if (p.ck) {  // the full pass of a training forward: y and the backward's checkpoints
      if (sp && z) return launch_chan_k<TY, N, true, true, false, false, true>(p, maps, nseg, st);
      if (sp) return launch_chan_k<TY, N, true, false, false, false, true>(p, maps, nseg, st);
      if (z) return launch_chan_k<TY, N, false, true, false, false, true>(p, maps, nseg, st);
      return launch_chan_k<TY, N, false, false, false, false, true>(p, maps, nseg, st);
    }
  }
  if (sp && z) return launch_chan_k<TY, N, true, !kAgg, kAgg, kConv>(p, maps, nseg, st);
  if (sp) return launch_chan_k<TY, N, true, false, kAgg, kConv>(p, maps, nseg, st);
  if (z) return launch_chan_k<TY, N, false, !kAgg, kAgg, kConv>(p, maps, nseg, st);
  return launch_chan_k<TY, N, false, false, kAgg, kConv>(p, maps, nseg, st);
}
template <typename TY, int N, bool kAgg>
cudaError_t launch_chan_sw(const FwdParams& p, const CUtensorMap* maps, int nseg, cudaStream_t st, bool sp, bool z) {
  return p.conv_w ? launch_chan_sz<TY, N, kAgg, true>(p, maps, nseg, st, sp, z)
                  : launch_chan_sz<TY, N, kAgg, false>(p, maps, nseg, st, sp, z);
}

template <typename TY, int N>
cudaError_t launch_chan(const FwdParams& p0, const SegPlan& plan, void* ws, cudaStream_t st, bool* launched) {
  *launched = false;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType ydt = sizeof(TY) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : bf;
  const uint64_t L = (uint64_t)p0.L, Bt = (uint64_t)p0.batch, D = (uint64_t)p0.D;
  CUtensorMap maps[6];  // u, delta, z, B, C, y
  if (!encode_3d(&maps[0], p0.u, bf, 2, D, L, Bt, ssm::kChanCTA, kChanTC) ||
      !encode_3d(&maps[1], p0.delta, bf, 2, D, L, Bt, ssm::kChanCTA, kChanTC) ||
      !encode_3d(&maps[3], p0.B, bf, 2, N, L, Bt, N, kChanTC) ||
      !encode_3d(&maps[4], p0.C, bf, 2, N, L, Bt, N, kChanTC) ||
      !encode_3d(&maps[5], p0.y, ydt, sizeof(TY), D, L, Bt, 32, kChanTC))
    return cudaSuccess;
  if (p0.z) {
    if (!encode_3d(&maps[2], p0.z, bf, 2, D, L, Bt, ssm::kChanCTA, kChanTC)) return cudaSuccess;
  } else {
    maps[2] = maps[0];  // never read when there is no gate
  }
  *launched = true;
  const bool sp = p0.delta_softplus != 0, z = p0.z != nullptr;
  FwdParams p = p0;
  p.seg_len = p0.L;
  p.seg_h0 = p0.h0;  // one segment: the caller's start state (or zeros)
  p.seg_E = p.seg_P = nullptr;
  int nseg = 1;
  if (plan.nseg > 1 && !ws) {
    // No workspace: the segment values live in y itself (SegY), each in its channel's
    // column of its segment's first rows, until the full pass overwrites them.
    nseg = plan.nseg;
    p.seg_len = plan.seg_len;
    p.seg_h0 = nullptr;
    p.seg_y = p0.y;
    p.seg_y_bf16 = sizeof(TY) == 2 ? 1 : 0;
    FwdParams pa = p;
    pa.ck = nullptr;  // the aggregate pass starts every segment from zero: no checkpoints
    cudaError_t e = launch_chan_sw<__nv_bfloat16, N, true>(pa, maps, nseg - 1, st, sp, false);
    if (e != cudaSuccess) return e;
    const ssm::SegY sy{p0.y, p.seg_y_bf16, p0.L, p0.D, plan.seg_len, N};
    e = launch_carry(sy, nullptr, nullptr, p0.h0, nullptr, nseg, p0.batch * p0.D * N, st);
    if (e != cudaSuccess) return e;
  } else if (plan.nseg > 1 && ws) {
    // 1) aggregate pass over segments 0 .. nseg-2; 2) carry scan; 3) full pass.
    const int64_t stride = (int64_t)plan.nseg * p0.batch * p0.D * N;
    float* E = static_cast<float*>(ws);
    float* P = E + stride;
    float* H = P + stride;
    nseg = plan.nseg;
    p.seg_len = plan.seg_len;
    p.seg_h0 = nullptr;  // the aggregate pass runs every segment from zero; h0 enters in the carry scan
    p.seg_E = E;
    p.seg_P = P;
    FwdParams pa = p;
    pa.ck = nullptr;
    cudaError_t e = launch_chan_sw<__nv_bfloat16, N, true>(pa, maps, nseg - 1, st, sp, false);
    if (e != cudaSuccess) return e;
    e = launch_carry(ssm::SegY{}, E, P, p0.h0, H, nseg, p0.batch * p0.D * N, st);
    if (e != cudaSuccess) return e;
    p.seg_h0 = H;
    p.seg_E = p.seg_P = nullptr;
  }
  return launch_chan_sw<TY, N, false>(p, maps, nseg, st, sp, z);
}

template <typename TY>
cudaError_t launch_chan_n(int64_t N, const FwdParams& p, const SegPlan& plan, void* ws, cudaStream_t st,
                          bool* launched) {
  if (N == 8) return launch_chan<TY, 8>(p, plan, ws, st, launched);
  return launch_chan<TY, 16>(p, plan, ws, st, launched);
}

// Checkpoints for the backward pass: the channel kernel's aggregate pass over one
// segment (the recurrence without read-out) writes the state before every kCkSteps-step
// chunk to ck[b][c][D][N]. *launched = false when a tensor map cannot be built.
template <int N>
cudaError_t launch_chan_ckpt(const FwdParams& p0, float* ck, int64_t nc, cudaStream_t st, bool* launched) {
  *launched = false;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t L = (uint64_t)p0.L, Bt = (uint64_t)p0.batch, D = (uint64_t)p0.D;
  CUtensorMap maps[6];  // u, delta, z, B, C, y
  if (!encode_3d(&maps[0], p0.u, bf, 2, D, L, Bt, ssm::kChanCTA, kChanTC) ||
      !encode_3d(&maps[1], p0.delta, bf, 2, D, L, Bt, ssm::kChanCTA, kChanTC) ||
      !encode_3d(&maps[3], p0.B, bf, 2, N, L, Bt, N, kChanTC))
    return cudaSuccess;
  maps[2] = maps[0];  // z, C and y: the aggregate pass reads and writes none of them
  maps[4] = maps[3];
  maps[5] = maps[0];
  *launched = true;
  FwdParams p = p0;
  p.seg_len = p0.L;
  p.seg_h0 = p0.h0;
  p.seg_E = p.seg_P = nullptr;
  p.seg_y = nullptr;
  p.ck = ck;
  p.ck_nc = nc;
  return launch_chan_sw<__nv_bfloat16, N, true>(p, maps, 1, st, p0.delta_softplus != 0, false);
}

// ---- generic forward launch ------------------------------------------------------------
constexpr int kGenDT = 32, kGenTC = 32;

// Segments for the generic kernel (32 channels per CTA) when its channel blocks cannot
// fill the GPU: at most 128 segments (the carry scan's four warps), each at least two chunks
// long and long enough to hold its carries in y (`rows` rows).
SegPlan plan_generic_segments(int64_t batch, int64_t L, int64_t D, int64_t rows) {
  SegPlan sp;
  sp.seg_len = L;
  const int sms = num_sms();
  const int64_t ctas = ((D + kGenDT - 1) / kGenDT) * batch;
  if (sms <= 0 || ctas <= 0 || ctas * 2 > sms) return sp;
  int64_t nseg = sms / ctas;
  if (nseg > 128) nseg = 128;
  const int64_t min_len = ((rows > 2 * kGenTC ? rows : 2 * kGenTC) + kGenTC - 1) / kGenTC * kGenTC;
  int64_t len = L;
  nseg = fit_segments(L, nseg, kGenTC, min_len, rows, &len);
  if (nseg < 2) return sp;
  sp.nseg = (int)nseg;
  sp.seg_len = len;
  return sp;
}

template <typename T, typename TY, int N, bool kAgg>
cudaError_t launch_fwd(const FwdParams& p, int nseg, cudaStream_t st) {
  constexpr int SPL = 4;
  dim3 grid((unsigned)((p.D + kGenDT - 1) / kGenDT), (unsigned)p.batch, (unsigned)nseg);
  dim3 block(kGenDT * (N / SPL));
  void* args[] = {const_cast<FwdParams*>(&p)};
  const void* kern =
      p.zoh ? reinterpret_cast<const void*>(&ssm::scan_fwd_generic<T, TY, N, SPL, kGenDT, kGenTC, true, kAgg>)
            : reinterpret_cast<const void*>(&ssm::scan_fwd_generic<T, TY, N, SPL, kGenDT, kGenTC, false, kAgg>);
  return cudaLaunchKernel(kern, grid, block, args, 0, st);
}

// One pass, or, when the channel blocks are too few, the segmented schedule with its
// carries in y: aggregate pass over segments 0 .. nseg-2, carry scan, full pass.
template <typename T, typename TY, int N>
cudaError_t launch_fwd_seg(const FwdParams& p0, cudaStream_t st) {
  const SegPlan plan = plan_generic_segments(p0.batch, p0.L, p0.D, (sizeof(TY) == 2 ? 6 : 3) * N);
  if (plan.nseg <= 1) return launch_fwd<T, TY, N, false>(p0, 1, st);
  FwdParams p = p0;
  p.seg_y = p0.y;
  p.seg_y_bf16 = sizeof(TY) == 2 ? 1 : 0;
  p.seg_len = plan.seg_len;
  int nseg = plan.nseg;
  cudaError_t e = launch_fwd<T, TY, N, true>(p, nseg - 1, st);
  if (e != cudaSuccess) return e;
  const ssm::SegY sy{p0.y, p.seg_y_bf16, p0.L, p0.D, plan.seg_len, N};
  e = launch_carry(sy, nullptr, nullptr, p0.h0, nullptr, nseg, p0.batch * p0.D * N, st);
  if (e != cudaSuccess) return e;
  return launch_fwd<T, TY, N, false>(p, nseg, st);
}

template <typename T, typename TY>
cudaError_t launch_fwd_n(int64_t N, const FwdParams& p, cudaStream_t st) {
  switch (N) {
    case 4: return launch_fwd_seg<T, TY, 4>(p, st);
    case 8: return launch_fwd_seg<T, TY, 8>(p, st);
    default: return launch_fwd_seg<T, TY, 16>(p, st);
  }
}

// ---- decode launch -------------------------------------------------------------------
// The streamed decode kernel: the plain step with bf16 inputs and N = 16 when D splits
// into whole tiles and every streamed tensor starts 16-byte aligned.
template <typename TY>
cudaError_t launch_dec_stream(const DecodeParams& p, cudaStream_t st, bool* launched) {
  *launched = false;
  if (p.zoh || p.D % ssm::kDecTile != 0) return cudaSuccess;
  for (const void* q : {static_cast<const void*>(p.state), p.x, p.delta, static_cast<const void*>(p.A), p.B, p.C, p.z,
                        static_cast<const void*>(p.delta_bias), static_cast<const void*>(p.conv_w),
                        static_cast<const void*>(p.conv_b), static_cast<const void*>(p.conv_state)})
    if (!aligned16(q)) return cudaSuccess;
  const bool map = p.delta_bias || p.delta_softplus, conv = p.conv_w != nullptr;
  auto kern = conv ? (map ? &ssm::state_update_stream<TY, true, true> : &ssm::state_update_stream<TY, false, true>)
                   : (map ? &ssm::state_update_stream<TY, true, false> : &ssm::state_update_stream<TY, false, false>);
  constexpr int smem = ssm::dec_stream_smem_bytes();
  constexpr int threads = ssm::kDecConsumers + 32;
  static const auto set_up = [](const void* k, int* per_sm) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, k, threads, smem);
    if (*per_sm < 1) *per_sm = 1;
    return e;
  };
  static int per_sm[4] = {0, 0, 0, 0};
  static const cudaError_t attr[4] = {
      set_up(reinterpret_cast<const void*>(&ssm::state_update_stream<TY, false, false>), &per_sm[0]),
      set_up(reinterpret_cast<const void*>(&ssm::state_update_stream<TY, true, false>), &per_sm[1]),
      set_up(reinterpret_cast<const void*>(&ssm::state_update_stream<TY, false, true>), &per_sm[2]),
      set_up(reinterpret_cast<const void*>(&ssm::state_update_stream<TY, true, true>), &per_sm[3])};
  const int vi = (map ? 1 : 0) + (conv ? 2 : 0);
  if (attr[vi] != cudaSuccess) return attr[vi];
  int64_t ntiles = p.batch * p.D / ssm::kDecTile;
  int64_t grid = (int64_t)(num_sms() > 0 ? num_sms() : 1) * per_sm[vi];
  if (grid > ntiles) grid = ntiles;
  *launched = true;
  long long wc = wait_limit_cycles();
  int skip = fault_skip_loads();
  void* args[] = {const_cast<DecodeParams*>(&p), &ntiles, &wc, &skip};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), dim3((unsigned)grid), dim3(threads), args, smem, st);
}

template <typename T, typename TY, int N>
cudaError_t launch_dec(const DecodeParams& p, cudaStream_t st) {
  if constexpr (N == 16 && sizeof(T) == 2) {
    if (decode_streamed()) {
      bool launched = false;
      const cudaError_t e = launch_dec_stream<TY>(p, st, &launched);
      if (e != cudaSuccess || launched) return e;
    }
  }
  const int64_t threads = p.batch * p.D * (N / (N >= 8 ? 8 : 4));  // 8 states per thread (4 for N = 4)
  dim3 grid((unsigned)((threads + 255) / 256)), block(256);
  void* args[] = {const_cast<DecodeParams*>(&p)};
  const bool ext = p.delta_bias || p.delta_softplus || p.zoh || p.conv_w;
  const void* kern = ext ? reinterpret_cast<const void*>(&ssm::state_update_kernel<T, TY, N, true>)
                         : reinterpret_cast<const void*>(&ssm::state_update_kernel<T, TY, N, false>);
  return cudaLaunchKernel(kern, grid, block, args, 0, st);
}

template <typename T, typename TY>
cudaError_t launch_dec_n(int64_t N, const DecodeParams& p, cudaStream_t st) {
  switch (N) {
    case 4: return launch_dec<T, TY, 4>(p, st);
    case 8: return launch_dec<T, TY, 8>(p, st);
    default: return launch_dec<T, TY, 16>(p, st);
  }
}

}  // namespace

extern "C" {

const char* ssm_status_string(ssm_status_t s) {
  switch (s) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_NULL: return "SSM_ERR_NULL: a required descriptor or data pointer is NULL";
    case SSM_ERR_SHAPE: return "SSM_ERR_SHAPE: ndim or a dimension does not match the contract";
    case SSM_ERR_DTYPE: return "SSM_ERR_DTYPE: element type not allowed or I/O types differ";
    case SSM_ERR_LAYOUT: return "SSM_ERR_LAYOUT: misaligned pointer or an output overlaps an input";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: request not implemented by this build";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA: the CUDA runtime reported an error";
    case SSM_ERR_DEVICE_TIMEOUT: return "SSM_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "SSM_ERR_UNKNOWN";
}

}  // extern "C"

namespace {

// The conv prologue's tensors (all null = no prologue).
struct ConvArgs {
  const ssm_tensor_t* w = nullptr;  // (D, 4) f32
  const ssm_tensor_t* b = nullptr;  // (D) f32, nullable
  ssm_tensor_t* state = nullptr;    // (batch, D, 3) I/O type, nullable: read, then overwritten
};

ssm_status_t check_conv(const ConvArgs* c, int64_t batch, int64_t Dm, ssm_dtype_t io) {
  ssm_status_t s;
  if ((s = check_tensor(c->w, {Dm, 4})) != SSM_OK) return s;
  if (c->b && (s = check_tensor(c->b, {Dm})) != SSM_OK) return s;
  if (c->state && (s = check_tensor(c->state, {batch, Dm, 3})) != SSM_OK) return s;
  if (c->w->dtype != SSM_F32 || (c->b && c->b->dtype != SSM_F32) || (c->state && c->state->dtype != io))
    return SSM_ERR_DTYPE;
  return SSM_OK;
}

// After the scan: the conv state moves on to the last three inputs (stream order puts
// this after every read of the old state).
ssm_status_t finish_fwd(cudaError_t e, const FwdParams& p, ssm_dtype_t io, ssm_tensor_t* conv_state, cudaStream_t st) {
  if (e == cudaSuccess && conv_state) {
    const int64_t n = p.batch * p.D;
    dim3 grid((unsigned)((n + 255) / 256)), block(256);
    int64_t batch = p.batch, L = p.L, D = p.D;
    const void* x = p.u;
    void* cs = conv_state->data;
    void* args[] = {&x, &cs, &batch, &L, &D};
    const void* kern = io == SSM_F32 ? reinterpret_cast<const void*>(&ssm::conv_state_next_kernel<float>)
                                     : reinterpret_cast<const void*>(&ssm::conv_state_next_kernel<__nv_bfloat16>);
    e = cudaLaunchKernel(kern, grid, block, args, 0, st);
  }
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// The backward pass's checkpoint region, for a training forward (written only by the
// channel kernel: *written = 1 when it ran).
struct CkArgs {
  float* ck;
  int64_t nc;
  int32_t* written;
};

ssm_status_t fwd_impl(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A, const ssm_tensor_t* B,
                      const ssm_tensor_t* C, const ssm_tensor_t* D, const ssm_tensor_t* z,
                      const ssm_tensor_t* delta_bias, int delta_softplus, const ssm_tensor_t* h0, uint32_t flags,
                      ssm_tensor_t* y, ssm_tensor_t* last_state, void* workspace, size_t workspace_bytes,
                      void* stream, const ConvArgs* conv = nullptr, const CkArgs* ck = nullptr) {
  if (!u || !delta || !A || !B || !C || !y) return SSM_ERR_NULL;
  if (u->ndim != 3 || A->ndim != 2) return SSM_ERR_SHAPE;
  const int64_t batch = u->shape[0], L = u->shape[1], Dm = u->shape[2], N = A->shape[1];
  if (batch < 0 || L < 0 || Dm < 0 || N < 0) return SSM_ERR_SHAPE;
  ssm_status_t s;
  if ((s = check_tensor(u, {batch, L, Dm})) != SSM_OK) return s;
  if ((s = check_tensor(delta, {batch, L, Dm})) != SSM_OK) return s;
  if ((s = check_tensor(A, {Dm, N})) != SSM_OK) return s;
  if ((s = check_tensor(B, {batch, L, N})) != SSM_OK) return s;
  if ((s = check_tensor(C, {batch, L, N})) != SSM_OK) return s;
  if (D && (s = check_tensor(D, {Dm})) != SSM_OK) return s;
  if (z && (s = check_tensor(z, {batch, L, Dm})) != SSM_OK) return s;
  if (delta_bias && (s = check_tensor(delta_bias, {Dm})) != SSM_OK) return s;
  if ((s = check_tensor(y, {batch, L, Dm})) != SSM_OK) return s;
  if (last_state && (s = check_tensor(last_state, {batch, Dm, N})) != SSM_OK) return s;
  if (h0 && (s = check_tensor(h0, {batch, Dm, N})) != SSM_OK) return s;

  const ssm_dtype_t io = u->dtype;
  if (delta->dtype != io || B->dtype != io || C->dtype != io || (z && z->dtype != io)) return SSM_ERR_DTYPE;
  if (y->dtype != io && y->dtype != SSM_F32) return SSM_ERR_DTYPE;
  if (A->dtype != SSM_F32 || (D && D->dtype != SSM_F32) || (delta_bias && delta_bias->dtype != SSM_F32) ||
      (last_state && last_state->dtype != SSM_F32) || (h0 && h0->dtype != SSM_F32))
    return SSM_ERR_DTYPE;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_UNSUPPORTED;
  if ((flags & ~SSM_FWD_ZOH) != 0) return SSM_ERR_UNSUPPORTED;
  if (!n_supported(N)) return SSM_ERR_UNSUPPORTED;
  if (batch > 65535) return SSM_ERR_UNSUPPORTED;

  if (conv && (s = check_conv(conv, batch, Dm, io)) != SSM_OK) return s;
  const ssm_tensor_t* cw = conv ? conv->w : nullptr;
  const ssm_tensor_t* cb = conv ? conv->b : nullptr;
  ssm_tensor_t* cst = conv ? conv->state : nullptr;
  if (cst) {  // in/out: it may overlap nothing else
    const ssm_tensor_t* all[] = {u, delta, A, B, C, D, z, delta_bias, h0, y, last_state, cw, cb};
    for (const ssm_tensor_t* t : all)
      if (overlaps(cst, t)) return SSM_ERR_LAYOUT;
  }

  const ssm_tensor_t* ins[] = {u, delta, A, B, C, D, z, delta_bias, h0, cw, cb};
  // last_state may be exactly the h0 buffer (read first, then overwritten by the same thread).
  const bool state_in_place = h0 && last_state && h0->data == last_state->data;
  for (const ssm_tensor_t* in : ins) {
    if (overlaps(y, in)) return SSM_ERR_LAYOUT;
    if (last_state && !(state_in_place && in == h0) && overlaps(last_state, in)) return SSM_ERR_LAYOUT;
  }
  if (last_state && overlaps(last_state, y)) return SSM_ERR_LAYOUT;
  if (workspace && workspace_bytes > 0) {
    ssm_tensor_t w{};
    w.data = workspace;
    w.dtype = SSM_F32;
    w.ndim = 1;
    w.shape[0] = (int64_t)(workspace_bytes / 4);
    const ssm_tensor_t* all[] = {u, delta, A, B, C, D, z, delta_bias, h0, y, last_state, cw, cb, cst};
    for (const ssm_tensor_t* t : all)
      if (overlaps(&w, t)) return SSM_ERR_LAYOUT;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (batch == 0 || Dm == 0) return SSM_OK;
  if (L == 0) {  // the state is unchanged: h0, or zeros
    if (last_state && !state_in_place) {
      const size_t bytes = (size_t)(numel(last_state) * 4);
      const cudaError_t e = h0 ? cudaMemcpyAsync(last_state->data, h0->data, bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(last_state->data, 0, bytes, st);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }

  FwdParams p;
  p.u = u->data;
  p.delta = delta->data;
  p.A = static_cast<const float*>(A->data);
  p.B = B->data;
  p.C = C->data;
  p.Dskip = D ? static_cast<const float*>(D->data) : nullptr;
  p.z = z ? z->data : nullptr;
  p.delta_bias = delta_bias ? static_cast<const float*>(delta_bias->data) : nullptr;
  p.delta_softplus = delta_softplus;
  p.y = y->data;
  p.last_state = last_state ? static_cast<float*>(last_state->data) : nullptr;
  p.h0 = h0 ? static_cast<const float*>(h0->data) : nullptr;
  p.zoh = (flags & SSM_FWD_ZOH) ? 1 : 0;
  p.conv_w = cw ? static_cast<const float*>(cw->data) : nullptr;
  p.conv_b = cb ? static_cast<const float*>(cb->data) : nullptr;
  p.conv_state = cst ? cst->data : nullptr;
  p.batch = batch;
  p.L = L;
  p.D = Dm;

  p.seg_len = L;
  p.seg_h0 = nullptr;
  p.seg_E = p.seg_P = nullptr;
  p.seg_y = nullptr;
  p.seg_y_bf16 = 0;
  p.wait_cycles = wait_limit_cycles();
  p.fault_skip_loads = fault_skip_loads();
  p.ck = ck ? ck->ck : nullptr;
  p.ck_nc = ck ? ck->nc : 0;

  cudaError_t e;
  const FwdVariant var = forward_variant();
  if (io == SSM_BF16 && var != FwdVariant::kGeneric && chan_eligible(p, N)) {
    SegPlan plan = plan_segments(batch, L, Dm, N);
    const bool use_ws = plan.nseg > 1 && workspace && workspace_bytes >= plan.bytes &&
                        reinterpret_cast<uintptr_t>(workspace) % 16 == 0;
    // Without a (large enough) workspace the segments keep their values in y, which needs
    // 6 N rows per segment (3 N for fp32 y); otherwise one segment.
    const int64_t rows = (y->dtype == SSM_BF16 ? 6 : 3) * N;
    if (!use_ws && (plan.nseg <= 1 || plan.seg_len < rows)) plan = SegPlan{1, L, 0};
    bool launched = false;
    e = y->dtype == SSM_BF16 ? launch_chan_n<__nv_bfloat16>(N, p, plan, use_ws ? workspace : nullptr, st, &launched)
                             : launch_chan_n<float>(N, p, plan, use_ws ? workspace : nullptr, st, &launched);
    if (ck && launched && e == cudaSuccess) *ck->written = 1;
    if (launched || e != cudaSuccess) return finish_fwd(e, p, io, cst, st);
  }
  if (io == SSM_F32)
    e = launch_fwd_n<float, float>(N, p, st);
  else if (y->dtype == SSM_BF16)
    e = launch_fwd_n<__nv_bfloat16, __nv_bfloat16>(N, p, st);
  else
    e = launch_fwd_n<__nv_bfloat16, float>(N, p, st);
  return finish_fwd(e, p, io, cst, st);
}

}  // namespace

extern "C" {

ssm_status_t ssm_selective_scan_fwd(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                    const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                    const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                    ssm_tensor_t* y, ssm_tensor_t* last_state, void* stream) {
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, 0u, y, last_state, nullptr, 0, stream);
}

ssm_status_t ssm_selective_scan_fwd_workspace_size(int64_t batch, int64_t L, int64_t D, int64_t N, size_t* bytes) {
  if (!bytes) return SSM_ERR_NULL;
  if (batch < 0 || L < 0 || D < 0 || N < 0) return SSM_ERR_SHAPE;
  *bytes = 0;
  if (batch == 0 || L == 0 || D == 0 || !n_supported(N)) return SSM_OK;
  *bytes = plan_segments(batch, L, D, N).bytes;
  return SSM_OK;
}

ssm_status_t ssm_selective_scan_fwd_ws(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                       const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                       const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                       ssm_tensor_t* y, ssm_tensor_t* last_state, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (workspace_bytes > 0 && !workspace) return SSM_ERR_NULL;
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SSM_ERR_LAYOUT;
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, 0u, y, last_state, workspace, workspace_bytes,
                  stream);
}

ssm_status_t ssm_selective_scan_fwd_ex(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                       const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                       const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                       const ssm_tensor_t* h0, uint32_t flags, ssm_tensor_t* y,
                                       ssm_tensor_t* last_state, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (workspace_bytes > 0 && !workspace) return SSM_ERR_NULL;
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SSM_ERR_LAYOUT;
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, flags, y, last_state, workspace,
                  workspace_bytes, stream);
}

namespace {
ssm_status_t dec_impl(ssm_tensor_t* state, const ssm_tensor_t* x, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                      const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D, const ssm_tensor_t* z,
                      const ssm_tensor_t* delta_bias, int delta_softplus, uint32_t flags, ssm_tensor_t* y,
                      void* stream, const ConvArgs* conv = nullptr) {
  if (!state || !x || !delta || !A || !B || !C || !y) return SSM_ERR_NULL;
  if (conv && (!conv->w || !conv->state)) return SSM_ERR_NULL;
  if (state->ndim != 3) return SSM_ERR_SHAPE;
  const int64_t batch = state->shape[0], Dm = state->shape[1], N = state->shape[2];
  if (batch < 0 || Dm < 0 || N < 0) return SSM_ERR_SHAPE;
  ssm_status_t s;
  if ((s = check_tensor(state, {batch, Dm, N}, true)) != SSM_OK) return s;
  if ((s = check_tensor(x, {batch, Dm})) != SSM_OK) return s;
  if ((s = check_tensor(delta, {batch, Dm})) != SSM_OK) return s;
  if ((s = check_tensor(A, {Dm, N}, true)) != SSM_OK) return s;
  if ((s = check_tensor(B, {batch, N})) != SSM_OK) return s;
  if ((s = check_tensor(C, {batch, N})) != SSM_OK) return s;
  if (D && (s = check_tensor(D, {Dm})) != SSM_OK) return s;
  if (z && (s = check_tensor(z, {batch, Dm})) != SSM_OK) return s;
  if ((s = check_tensor(y, {batch, Dm})) != SSM_OK) return s;
  if (delta_bias && (s = check_tensor(delta_bias, {Dm})) != SSM_OK) return s;

  const ssm_dtype_t io = x->dtype;
  if (delta->dtype != io || B->dtype != io || C->dtype != io || (z && z->dtype != io)) return SSM_ERR_DTYPE;
  if (y->dtype != io && y->dtype != SSM_F32) return SSM_ERR_DTYPE;
  if (state->dtype != SSM_F32 || A->dtype != SSM_F32 || (D && D->dtype != SSM_F32) ||
      (delta_bias && delta_bias->dtype != SSM_F32))
    return SSM_ERR_DTYPE;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_UNSUPPORTED;
  if ((flags & ~SSM_FWD_ZOH) != 0) return SSM_ERR_UNSUPPORTED;
  if (!n_supported(N)) return SSM_ERR_UNSUPPORTED;

  if (conv && (s = check_conv(conv, batch, Dm, io)) != SSM_OK) return s;
  const ssm_tensor_t* cw = conv ? conv->w : nullptr;
  const ssm_tensor_t* cb = conv ? conv->b : nullptr;
  ssm_tensor_t* cst = conv ? conv->state : nullptr;
  const ssm_tensor_t* ins[] = {x, delta, A, B, C, D, z, delta_bias, cw, cb};
  for (const ssm_tensor_t* in : ins) {
    if (overlaps(y, in)) return SSM_ERR_LAYOUT;
    if (overlaps(state, in)) return SSM_ERR_LAYOUT;
    if (cst && overlaps(cst, in)) return SSM_ERR_LAYOUT;
  }
  if (overlaps(state, y)) return SSM_ERR_LAYOUT;
  if (cst && (overlaps(cst, y) || overlaps(cst, state))) return SSM_ERR_LAYOUT;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (batch == 0 || Dm == 0) return SSM_OK;

  DecodeParams p;
  p.state = static_cast<float*>(state->data);
  p.x = x->data;
  p.delta = delta->data;
  p.A = static_cast<const float*>(A->data);
  p.B = B->data;
  p.C = C->data;
  p.Dskip = D ? static_cast<const float*>(D->data) : nullptr;
  p.z = z ? z->data : nullptr;
  p.y = y->data;
  p.delta_bias = delta_bias ? static_cast<const float*>(delta_bias->data) : nullptr;
  p.delta_softplus = delta_softplus;
  p.zoh = (flags & SSM_FWD_ZOH) ? 1 : 0;
  p.conv_w = cw ? static_cast<const float*>(cw->data) : nullptr;
  p.conv_b = cb ? static_cast<const float*>(cb->data) : nullptr;
  p.conv_state = cst ? cst->data : nullptr;
  p.batch = batch;
  p.D = Dm;

  cudaError_t e;
  if (io == SSM_F32)
    e = launch_dec_n<float, float>(N, p, st);
  else if (y->dtype == SSM_BF16)
    e = launch_dec_n<__nv_bfloat16, __nv_bfloat16>(N, p, st);
  else
    e = launch_dec_n<__nv_bfloat16, float>(N, p, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
}  // namespace

ssm_status_t ssm_state_update(ssm_tensor_t* state, const ssm_tensor_t* x, const ssm_tensor_t* delta,
                              const ssm_tensor_t* A, const ssm_tensor_t* B, const ssm_tensor_t* C,
                              const ssm_tensor_t* D, const ssm_tensor_t* z, ssm_tensor_t* y, void* stream) {
  return dec_impl(state, x, delta, A, B, C, D, z, nullptr, 0, 0u, y, stream);
}

ssm_status_t ssm_state_update_ex(ssm_tensor_t* state, const ssm_tensor_t* x, const ssm_tensor_t* delta,
                                 const ssm_tensor_t* A, const ssm_tensor_t* B, const ssm_tensor_t* C,
                                 const ssm_tensor_t* D, const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                 int delta_softplus, uint32_t flags, ssm_tensor_t* y, void* stream) {
  return dec_impl(state, x, delta, A, B, C, D, z, delta_bias, delta_softplus, flags, y, stream);
}

ssm_status_t ssm_conv_selective_scan_fwd(const ssm_tensor_t* x, const ssm_tensor_t* conv_weight,
                                         const ssm_tensor_t* conv_bias, ssm_tensor_t* conv_state,
                                         const ssm_tensor_t* delta, const ssm_tensor_t* A, const ssm_tensor_t* B,
                                         const ssm_tensor_t* C, const ssm_tensor_t* D, const ssm_tensor_t* z,
                                         const ssm_tensor_t* delta_bias, int delta_softplus, const ssm_tensor_t* h0,
                                         uint32_t flags, ssm_tensor_t* y, ssm_tensor_t* last_state, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (!conv_weight) return SSM_ERR_NULL;
  if (workspace_bytes > 0 && !workspace) return SSM_ERR_NULL;
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SSM_ERR_LAYOUT;
  ConvArgs c;
  c.w = conv_weight;
  c.b = conv_bias;
  c.state = conv_state;
  return fwd_impl(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, flags, y, last_state, workspace,
                  workspace_bytes, stream, &c);
}

ssm_status_t ssm_conv_state_update(ssm_tensor_t* conv_state, ssm_tensor_t* state, const ssm_tensor_t* x,
                                   const ssm_tensor_t* conv_weight, const ssm_tensor_t* conv_bias,
                                   const ssm_tensor_t* delta, const ssm_tensor_t* A, const ssm_tensor_t* B,
                                   const ssm_tensor_t* C, const ssm_tensor_t* D, const ssm_tensor_t* z,
                                   const ssm_tensor_t* delta_bias, int delta_softplus, uint32_t flags,
                                   ssm_tensor_t* y, void* stream) {
  ConvArgs c;
  c.w = conv_weight;
  c.b = conv_bias;
  c.state = conv_state;
  return dec_impl(state, x, delta, A, B, C, D, z, delta_bias, delta_softplus, flags, y, stream, &c);
}

}  // extern "C"

namespace {
// ---- backward pass -------------------------------------------------------------------
struct BwdPlan {
  int nc = 0, W = 0;
  size_t off_ck = 0, off_part = 0, off_dA = 0, off_dD = 0, off_db = 0, bytes = 0;
};
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
BwdPlan plan_bwd(int64_t batch, int64_t L, int64_t D, int64_t N) {
  BwdPlan pl;
  pl.nc = (int)((L + ssm::kBwdK - 1) / ssm::kBwdK);
  pl.W = (int)((D + ssm::kBwdCh - 1) / ssm::kBwdCh);
  size_t o = 0;
  pl.off_ck = o;
  o += round256((size_t)batch * pl.nc * D * N * 4);
  pl.off_part = o;
  o += round256((size_t)batch * L * pl.W * 2 * N * 4);
  pl.off_dA = o;
  o += round256((size_t)batch * D * N * 4);
  pl.off_dD = o;
  o += round256((size_t)batch * D * 4);
  pl.off_db = o;
  o += round256((size_t)batch * D * 4);
  pl.bytes = o;
  return pl;
}

template <typename T, typename TG, int N>
cudaError_t launch_bwd(const ssm::BwdParams& p, cudaStream_t st) {
  auto kern = &ssm::scan_bwd_kernel<T, TG, N>;
  constexpr int smem = ssm::bwd_smem_bytes<T, TG, N>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  void* args[] = {const_cast<ssm::BwdParams*>(&p)};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kern), dim3((unsigned)p.W, (unsigned)p.batch), dim3(32), args,
                          smem, st);
}

template <typename T, typename TG>
cudaError_t launch_bwd_n(int64_t N, const ssm::BwdParams& p, cudaStream_t st) {
  switch (N) {
    case 4: return launch_bwd<T, TG, 4>(p, st);
    case 8: return launch_bwd<T, TG, 8>(p, st);
    default: return launch_bwd<T, TG, 16>(p, st);
  }
}

template <typename TG>
cudaError_t launch_bwd_reduce(const ssm::BwdParams& p, int64_t N, void* dB, void* dC, float* dA, float* dD,
                              float* dbias, cudaStream_t st) {
  const int64_t n = p.batch * p.L * N + p.D * N + p.D;
  const float* part = p.part;
  const float* dAp = p.dA_part;
  const float* dDp = p.dD_part;
  const float* dbp = p.dbias_part;
  TG* b = static_cast<TG*>(dB);
  TG* c = static_cast<TG*>(dC);
  int64_t batch = p.batch, L = p.L, D = p.D;
  int Ni = (int)N, W = p.W;
  void* args[] = {&part, &dAp, &dDp, &dbp, &b, &c, &dA, &dD, &dbias, &batch, &L, &D, &Ni, &W};
  return cudaLaunchKernel(reinterpret_cast<const void*>(&ssm::scan_bwd_reduce<TG>), dim3((unsigned)((n + 255) / 256)),
                          dim3(256), args, 0, st);
}
}  // namespace

extern "C" {

ssm_status_t ssm_selective_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t D, int64_t N, size_t* bytes) {
  if (!bytes) return SSM_ERR_NULL;
  if (batch < 0 || L < 0 || D < 0 || N < 0) return SSM_ERR_SHAPE;
  *bytes = 0;
  if (batch == 0 || L == 0 || D == 0 || !n_supported(N)) return SSM_OK;
  *bytes = plan_bwd(batch, L, D, N).bytes;
  return SSM_OK;
}

ssm_status_t ssm_selective_scan_bwd_ex(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                       const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                       const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                       const ssm_tensor_t* h0, const ssm_tensor_t* dy, const ssm_tensor_t* dlast,
                                       ssm_tensor_t* du, ssm_tensor_t* ddelta, ssm_tensor_t* dA, ssm_tensor_t* dB,
                                       ssm_tensor_t* dC, ssm_tensor_t* dD, ssm_tensor_t* dz, ssm_tensor_t* dbias,
                                       ssm_tensor_t* dh0, uint32_t flags, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (flags & ~SSM_BWD_CHECKPOINTS) return SSM_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC) return SSM_ERR_NULL;
  if ((D != nullptr) != (dD != nullptr) || (z != nullptr) != (dz != nullptr) ||
      (delta_bias != nullptr) != (dbias != nullptr))
    return SSM_ERR_NULL;  // a gradient output exactly for each optional input
  if (u->ndim != 3 || A->ndim != 2) return SSM_ERR_SHAPE;
  const int64_t batch = u->shape[0], L = u->shape[1], Dm = u->shape[2], N = A->shape[1];
  if (batch < 0 || L < 0 || Dm < 0 || N < 0) return SSM_ERR_SHAPE;
  ssm_status_t s;
  const std::initializer_list<int64_t> sLD = {batch, L, Dm}, sLN = {batch, L, N}, sDN3 = {batch, Dm, N};
  for (const ssm_tensor_t* t : {u, delta, dy, static_cast<const ssm_tensor_t*>(du),
                                static_cast<const ssm_tensor_t*>(ddelta)})
    if ((s = check_tensor(t, sLD)) != SSM_OK) return s;
  if (z && ((s = check_tensor(z, sLD)) != SSM_OK || (s = check_tensor(dz, sLD)) != SSM_OK)) return s;
  if ((s = check_tensor(A, {Dm, N})) != SSM_OK || (s = check_tensor(dA, {Dm, N})) != SSM_OK) return s;
  for (const ssm_tensor_t* t : {B, C, static_cast<const ssm_tensor_t*>(dB), static_cast<const ssm_tensor_t*>(dC)})
    if ((s = check_tensor(t, sLN)) != SSM_OK) return s;
  if (D && ((s = check_tensor(D, {Dm})) != SSM_OK || (s = check_tensor(dD, {Dm})) != SSM_OK)) return s;
  if (delta_bias && ((s = check_tensor(delta_bias, {Dm})) != SSM_OK || (s = check_tensor(dbias, {Dm})) != SSM_OK))
    return s;
  if (h0 && (s = check_tensor(h0, sDN3)) != SSM_OK) return s;
  if (dlast && (s = check_tensor(dlast, sDN3)) != SSM_OK) return s;
  if (dh0 && (s = check_tensor(dh0, sDN3)) != SSM_OK) return s;

  const ssm_dtype_t io = u->dtype, gt = du->dtype;
  if (delta->dtype != io || B->dtype != io || C->dtype != io || (z && z->dtype != io)) return SSM_ERR_DTYPE;
  if (gt != io && gt != SSM_F32) return SSM_ERR_DTYPE;
  if (dy->dtype != gt || ddelta->dtype != gt || dB->dtype != gt || dC->dtype != gt || (dz && dz->dtype != gt))
    return SSM_ERR_DTYPE;
  for (const ssm_tensor_t* t : {A, D, delta_bias, h0, dlast, static_cast<const ssm_tensor_t*>(dA),
                                static_cast<const ssm_tensor_t*>(dD), static_cast<const ssm_tensor_t*>(dbias),
                                static_cast<const ssm_tensor_t*>(dh0)})
    if (t && t->dtype != SSM_F32) return SSM_ERR_DTYPE;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_UNSUPPORTED;
  if (!n_supported(N)) return SSM_ERR_UNSUPPORTED;
  if (batch > 65535) return SSM_ERR_UNSUPPORTED;

  const ssm_tensor_t* ins[] = {u, delta, A, B, C, D, z, delta_bias, h0, dy, dlast};
  const ssm_tensor_t* outs[] = {du, ddelta, dA, dB, dC, dD, dz, dbias, dh0};
  for (const ssm_tensor_t* o : outs) {
    for (const ssm_tensor_t* in : ins)
      if (overlaps(o, in)) return SSM_ERR_LAYOUT;
    for (const ssm_tensor_t* o2 : outs)
      if (o != o2 && overlaps(o, o2)) return SSM_ERR_LAYOUT;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool empty = batch == 0 || L == 0 || Dm == 0;
  const BwdPlan pl = empty ? BwdPlan{} : plan_bwd(batch, L, Dm, N);
  if (!empty) {
    if (!workspace) return SSM_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SSM_ERR_LAYOUT;
    if (workspace_bytes < pl.bytes) return SSM_ERR_SHAPE;
    ssm_tensor_t w{};
    w.data = workspace;
    w.dtype = SSM_F32;
    w.ndim = 1;
    w.shape[0] = (int64_t)(workspace_bytes / 4);
    for (const ssm_tensor_t* t : ins)
      if (overlaps(&w, t)) return SSM_ERR_LAYOUT;
    for (const ssm_tensor_t* t : outs)
      if (overlaps(&w, t)) return SSM_ERR_LAYOUT;
  }

  if (empty) {  // no steps: the sums are zero and dL/dh0 is dlast
    auto zero = [&](ssm_tensor_t* t) {
      return !t || numel(t) == 0 || cudaMemsetAsync(t->data, 0, (size_t)(numel(t) * elem_size(t->dtype)), st) == cudaSuccess;
    };
    bool ok = zero(dA) && zero(dD) && zero(dbias);
    if (dh0 && numel(dh0) > 0)
      ok = ok && (dlast ? cudaMemcpyAsync(dh0->data, dlast->data, (size_t)numel(dh0) * 4, cudaMemcpyDeviceToDevice, st) ==
                              cudaSuccess
                        : zero(dh0));
    return ok ? SSM_OK : SSM_ERR_CUDA;
  }

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  ssm::BwdParams p;
  p.u = u->data;
  p.delta = delta->data;
  p.A = static_cast<const float*>(A->data);
  p.B = B->data;
  p.C = C->data;
  p.Dskip = D ? static_cast<const float*>(D->data) : nullptr;
  p.z = z ? z->data : nullptr;
  p.delta_bias = delta_bias ? static_cast<const float*>(delta_bias->data) : nullptr;
  p.delta_softplus = delta_softplus;
  p.h0 = h0 ? static_cast<const float*>(h0->data) : nullptr;
  p.dy = dy->data;
  p.dlast = dlast ? static_cast<const float*>(dlast->data) : nullptr;
  p.du = du->data;
  p.ddelta = ddelta->data;
  p.dz = dz ? dz->data : nullptr;
  p.dh0 = dh0 ? static_cast<float*>(dh0->data) : nullptr;
  p.ck = reinterpret_cast<float*>(ws + pl.off_ck);
  p.part = reinterpret_cast<float*>(ws + pl.off_part);
  p.dA_part = reinterpret_cast<float*>(ws + pl.off_dA);
  p.dD_part = reinterpret_cast<float*>(ws + pl.off_dD);
  p.dbias_part = reinterpret_cast<float*>(ws + pl.off_db);
  p.batch = batch;
  p.L = L;
  p.D = Dm;
  p.nc = pl.nc;
  p.W = pl.W;
  {  // cp.async staging needs every (batch, L, D) row and every chunk of B, C 16-byte aligned
    const int64_t es = io == SSM_F32 ? 4 : 2, gs = gt == SSM_F32 ? 4 : 2;
    bool ok = (Dm * es) % 16 == 0 && (Dm * gs) % 16 == 0 && (L * N * es) % 16 == 0;
    for (const ssm_tensor_t* t : {u, delta, B, C, z, dy})
      if (t && reinterpret_cast<uintptr_t>(t->data) % 16 != 0) ok = false;
    p.async_ok = ok;
  }

  cudaError_t e;
  p.ck_ready = (flags & SSM_BWD_CHECKPOINTS) ? 1 : 0;  // written by ssm_selective_scan_fwd_train
  if (!p.ck_ready && io == SSM_BF16 && (N == 8 || N == 16) && forward_variant() != FwdVariant::kGeneric) {
    // The checkpoints from the channel kernel (as the forward pass's fast path)
    FwdParams fp{};
    fp.u = u->data;
    fp.delta = delta->data;
    fp.A = p.A;
    fp.B = B->data;
    fp.C = C->data;
    fp.delta_bias = p.delta_bias;
    fp.delta_softplus = delta_softplus;
    fp.h0 = p.h0;
    fp.batch = batch;
    fp.L = L;
    fp.D = Dm;
    fp.wait_cycles = wait_limit_cycles();
    if (chan_eligible(fp, N)) {
      bool launched = false;
      e = N == 8 ? launch_chan_ckpt<8>(fp, p.ck, p.nc, st, &launched) : launch_chan_ckpt<16>(fp, p.ck, p.nc, st, &launched);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
      p.ck_ready = launched ? 1 : 0;
    }
  }
  if (io == SSM_F32)
    e = launch_bwd_n<float, float>(N, p, st);
  else if (gt == SSM_BF16)
    e = launch_bwd_n<__nv_bfloat16, __nv_bfloat16>(N, p, st);
  else
    e = launch_bwd_n<__nv_bfloat16, float>(N, p, st);
  if (e != cudaSuccess) return SSM_ERR_CUDA;
  float* dAp = static_cast<float*>(dA->data);
  float* dDp = dD ? static_cast<float*>(dD->data) : nullptr;
  float* dbp = dbias ? static_cast<float*>(dbias->data) : nullptr;
  e = gt == SSM_BF16 ? launch_bwd_reduce<__nv_bfloat16>(p, N, dB->data, dC->data, dAp, dDp, dbp, st)
                     : launch_bwd_reduce<float>(p, N, dB->data, dC->data, dAp, dDp, dbp, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status_t ssm_selective_scan_bwd(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                    const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                    const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                    const ssm_tensor_t* h0, const ssm_tensor_t* dy, const ssm_tensor_t* dlast,
                                    ssm_tensor_t* du, ssm_tensor_t* ddelta, ssm_tensor_t* dA, ssm_tensor_t* dB,
                                    ssm_tensor_t* dC, ssm_tensor_t* dD, ssm_tensor_t* dz, ssm_tensor_t* dbias,
                                    ssm_tensor_t* dh0, void* workspace, size_t workspace_bytes, void* stream) {
  return ssm_selective_scan_bwd_ex(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, dy, dlast, du, ddelta, dA,
                                   dB, dC, dD, dz, dbias, dh0, 0u, workspace, workspace_bytes, stream);
}

ssm_status_t ssm_selective_scan_fwd_train(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                          const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                          const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                          const ssm_tensor_t* h0, ssm_tensor_t* y, ssm_tensor_t* last_state,
                                          void* bwd_workspace, size_t bwd_workspace_bytes,
                                          int32_t* checkpoints_written, void* stream) {
  if (!checkpoints_written || !u || !A) return SSM_ERR_NULL;
  *checkpoints_written = 0;
  if (u->ndim != 3 || A->ndim != 2) return SSM_ERR_SHAPE;
  const int64_t batch = u->shape[0], L = u->shape[1], Dm = u->shape[2], N = A->shape[1];
  if (batch < 0 || L < 0 || Dm < 0 || N < 0) return SSM_ERR_SHAPE;
  const bool empty = batch == 0 || L == 0 || Dm == 0 || !n_supported(N);
  CkArgs ck{nullptr, 0, checkpoints_written};
  if (!empty) {
    const BwdPlan pl = plan_bwd(batch, L, Dm, N);
    if (!bwd_workspace) return SSM_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(bwd_workspace) % 256 != 0) return SSM_ERR_LAYOUT;
    if (bwd_workspace_bytes < pl.bytes) return SSM_ERR_SHAPE;
    ssm_tensor_t w{};
    w.data = bwd_workspace;
    w.dtype = SSM_F32;
    w.ndim = 1;
    w.shape[0] = (int64_t)(bwd_workspace_bytes / 4);
    for (const ssm_tensor_t* t : {u, delta, A, B, C, D, z, delta_bias, h0, static_cast<const ssm_tensor_t*>(y),
                                  static_cast<const ssm_tensor_t*>(last_state)})
      if (t && overlaps(&w, t)) return SSM_ERR_LAYOUT;
    ck.ck = reinterpret_cast<float*>(static_cast<unsigned char*>(bwd_workspace) + pl.off_ck);
    ck.nc = pl.nc;
  }
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, 0u, y, last_state, nullptr, 0, stream,
                  nullptr, empty ? nullptr : &ck);
}

}  // extern "C"

namespace {
// Workspace of the chunk-parallel SSD schedule: per (b, c, h) the chunk's state
// contribution (fp32 P x N) and entering state (bf16 P x N), and per (b, h, c) its decay.
struct SsdPlan {
  size_t off_H = 0, off_dt = 0, off_cs = 0, off_CB = 0, bytes = 0;
};
SsdPlan ssd_plan(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P, int64_t N) {
  SsdPlan pl;
  if (batch <= 0 || L <= 0 || H <= 0 || G <= 0 || P <= 0 || N <= 0) return pl;
  const size_t nc = (size_t)((L + ssm::kSsdQ - 1) / ssm::kSsdQ), items = (size_t)batch * nc * H;
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  pl.off_H = 0;
  pl.off_dt = r256(items * P * N * 2);
  pl.off_cs = pl.off_dt + r256(items * ssm::kSsdQ * 4);
  pl.off_CB = pl.off_cs + r256(items * ssm::kSsdQ * 4);
  pl.bytes = pl.off_CB + r256((size_t)batch * nc * G * ssm::kSsdQ * ssm::kSsdCBPitch * 4);
  return pl;
}

// Persistent grid: as many CTAs as fit on the GPU at once, at most one per item.
unsigned persistent_grid(const void* kern, int threads, int smem, int64_t items) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t n = (int64_t)(num_sms() > 0 ? num_sms() : 1) * per_sm;
  if (n > items) n = items;
  return (unsigned)(n > 0 ? n : 1);
}

template <int P, int N>
cudaError_t launch_ssd(const ssm::SsdParams& p, bool y_f32, cudaStream_t st) {
  constexpr int smem = ssm::ssd_smem_bytes<P, N>();
  const void* kern = y_f32 ? reinterpret_cast<const void*>(&ssm::ssd_fwd_kernel<P, N, float>)
                           : reinterpret_cast<const void*>(&ssm::ssd_fwd_kernel<P, N, __nv_bfloat16>);
  const cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  void* args[] = {const_cast<ssm::SsdParams*>(&p)};
  return cudaLaunchKernel(kern, dim3((unsigned)p.H, (unsigned)p.batch), dim3(ssm::kSsdThreads), args, smem, st);
}

// Tensor maps of the chunk-parallel schedule: x as (p, head, batch row x step) and C as
// (group column, batch row x step), both in 64 x 64 boxes with the 128-byte swizzle (the
// read-out's ldmatrix layout and the tcgen05 walk's X operand); B as (group column, batch
// row x step) in 32 x 64 boxes (the walk's raw B).
bool ssd_maps(const ssm::SsdParams& p, int64_t P, int64_t N, CUtensorMap* tm_x, CUtensorMap* tm_c, CUtensorMap* tm_b) {
  auto fn = encode_fn();
  if (!fn || (uint64_t)(p.batch * p.L) >= (1ull << 31)) return false;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t H = (uint64_t)p.H, GN = (uint64_t)(p.G * N), rows = (uint64_t)(p.batch * p.L);
  const cuuint32_t Q = (cuuint32_t)ssm::kSsdQ;
  {
    cuuint64_t dims[3] = {(uint64_t)P, H, rows};
    cuuint64_t strides[2] = {(uint64_t)P * 2, H * P * 2};
    cuuint32_t box[3] = {64, 1, Q};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(tm_x, bf, 3, const_cast<void*>(static_cast<const void*>(p.x)), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  cuuint64_t dims[2] = {GN, rows};
  cuuint64_t strides[1] = {GN * 2};
  cuuint32_t estr[2] = {1, 1};
  {
    cuuint32_t box[2] = {64, Q};
    if (fn(tm_c, bf, 2, const_cast<void*>(static_cast<const void*>(p.C)), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  {
    cuuint32_t box[2] = {(cuuint32_t)ssm::kSsdNB, Q};
    if (fn(tm_b, bf, 2, const_cast<void*>(static_cast<const void*>(p.B)), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int P, int N>
cudaError_t launch_ssd_chunked(const ssm::SsdParams& p, bool y_f32, cudaStream_t st) {
  void* args[] = {const_cast<ssm::SsdParams*>(&p)};
  {
    const cudaError_t e = cudaLaunchKernel(reinterpret_cast<const void*>(&ssm::ssd_prep_kernel<N>),
                                           dim3((unsigned)p.nc, (unsigned)p.batch), dim3(256), args, 0, st);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_x, tm_c, tm_b;
  if (!ssd_maps(p, P, N, &tm_x, &tm_c, &tm_b)) return launch_ssd<P, N>(p, y_f32, st);  // no TMA: one CTA per head
  if (P == ssm::kTcP) {  // the state walk on tcgen05, operands by TMA
    constexpr int smem = ssm::SsdTcWalk<N>::kBytes;
    const void* k = reinterpret_cast<const void*>(&ssm::ssd_state_walk_tc_kernel<N>);
    void* targs[] = {&tm_x, &tm_b, const_cast<ssm::SsdParams*>(&p)};
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaLaunchKernel(k, dim3(N / ssm::kSsdNB, (unsigned)p.H, (unsigned)p.batch), dim3(ssm::kTcThreads), targs,
                           smem, st);
    if (e != cudaSuccess) return e;
  } else {
    constexpr int smem = ssm::ssd_walk_smem_bytes<P>();
    const void* k = reinterpret_cast<const void*>(&ssm::ssd_state_walk_kernel<P, N>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaLaunchKernel(k, dim3(N / ssm::kSsdNB, (unsigned)p.H, (unsigned)p.batch), dim3(ssm::kSsdThreads), args,
                           smem, st);
    if (e != cudaSuccess) return e;
  }
  void* sargs[] = {&tm_x, &tm_c, const_cast<ssm::SsdParams*>(&p)};
  const int64_t items = p.batch * p.nc * p.H;
  if (P == ssm::kTcP) {  // the read-out on tcgen05
    constexpr int smem = ssm::SsdTcScan<N>::kBytes;
    const void* k = y_f32 ? reinterpret_cast<const void*>(&ssm::ssd_chunk_scan_tc_kernel<N, float>)
                          : reinterpret_cast<const void*>(&ssm::ssd_chunk_scan_tc_kernel<N, __nv_bfloat16>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaLaunchKernel(k, dim3(persistent_grid(k, ssm::kTcScanThreads, smem, items)), dim3(ssm::kTcScanThreads),
                           sargs, smem, st);
    return e;
  }
  constexpr int smem = ssm::ssd_scan_smem_bytes<P, N>();
  const void* k = y_f32 ? reinterpret_cast<const void*>(&ssm::ssd_chunk_scan_kernel<P, N, float>)
                        : reinterpret_cast<const void*>(&ssm::ssd_chunk_scan_kernel<P, N, __nv_bfloat16>);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaLaunchKernel(k, dim3(persistent_grid(k, ssm::kSsdThreads, smem, items)), dim3(ssm::kSsdThreads), sargs,
                         smem, st);
  return e;
}

}  // namespace

extern "C" {

ssm_status_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t H, int64_t groups, int64_t P, int64_t N,
                                        size_t* bytes) {
  if (!bytes) return SSM_ERR_NULL;
  if (batch < 0 || L < 0 || H < 0 || groups < 1 || P < 0 || N < 0) return SSM_ERR_SHAPE;
  *bytes = ssd_plan(batch, L, H, groups, P, N).bytes;
  return SSM_OK;
}

ssm_status_t ssm_ssd_fwd(int64_t groups, const ssm_tensor_t* x, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                         const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                         const ssm_tensor_t* dt_bias, int dt_softplus, const ssm_tensor_t* h0, ssm_tensor_t* y,
                         ssm_tensor_t* last_state, void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace_bytes > 0 && !workspace) return SSM_ERR_NULL;
  if (!x || !delta || !A || !B || !C || !y) return SSM_ERR_NULL;
  if (x->ndim != 3 || A->ndim != 1 || B->ndim != 3) return SSM_ERR_SHAPE;
  const int64_t batch = x->shape[0], L = x->shape[1], HP = x->shape[2], H = A->shape[0], GN = B->shape[2];
  if (batch < 0 || L < 0 || HP < 0 || H <= 0 || groups <= 0 || H % groups != 0 || HP % H != 0 || GN % groups != 0)
    return SSM_ERR_SHAPE;
  const int64_t P = HP / H, N = GN / groups;
  ssm_status_t s;
  if ((s = check_tensor(x, {batch, L, HP})) != SSM_OK) return s;
  if ((s = check_tensor(delta, {batch, L, H})) != SSM_OK) return s;
  if ((s = check_tensor(A, {H})) != SSM_OK) return s;
  if ((s = check_tensor(B, {batch, L, GN})) != SSM_OK) return s;
  if ((s = check_tensor(C, {batch, L, GN})) != SSM_OK) return s;
  if (D && (s = check_tensor(D, {H})) != SSM_OK) return s;
  if (dt_bias && (s = check_tensor(dt_bias, {H})) != SSM_OK) return s;
  if (h0 && (s = check_tensor(h0, {batch, H, P * N})) != SSM_OK) return s;
  if ((s = check_tensor(y, {batch, L, HP})) != SSM_OK) return s;
  if (last_state && (s = check_tensor(last_state, {batch, H, P * N})) != SSM_OK) return s;
  if (x->dtype != SSM_BF16 || delta->dtype != SSM_BF16 || B->dtype != SSM_BF16 || C->dtype != SSM_BF16)
    return SSM_ERR_DTYPE;
  if (y->dtype != SSM_BF16 && y->dtype != SSM_F32) return SSM_ERR_DTYPE;
  for (const ssm_tensor_t* t : {A, D, dt_bias, h0, static_cast<const ssm_tensor_t*>(last_state)})
    if (t && t->dtype != SSM_F32) return SSM_ERR_DTYPE;
  if (dt_softplus != 0 && dt_softplus != 1) return SSM_ERR_UNSUPPORTED;
  if ((P != 64 && P != 128) || (N != 64 && N != 128) || batch > 65535 || H > INT32_MAX) return SSM_ERR_UNSUPPORTED;
  for (const ssm_tensor_t* t : {x, B, C})  // 16-byte vector loads
    if (numel(t) > 0 && reinterpret_cast<uintptr_t>(t->data) % 16 != 0) return SSM_ERR_LAYOUT;
  const ssm_tensor_t* ins[] = {x, delta, A, B, C, D, dt_bias, h0};
  for (const ssm_tensor_t* in : ins) {
    if (overlaps(y, in)) return SSM_ERR_LAYOUT;
    if (last_state && overlaps(last_state, in)) return SSM_ERR_LAYOUT;
  }
  if (last_state && overlaps(last_state, y)) return SSM_ERR_LAYOUT;
  const SsdPlan plan = ssd_plan(batch, L, H, groups, P, N);
  // (the chunk-parallel read-out walks its items with 32-bit counters: fewer than 2^31 items)
  const bool chunked = workspace && workspace_bytes >= plan.bytes && plan.bytes > 0 && H <= 65535 &&
                       batch * ((L + ssm::kSsdQ - 1) / ssm::kSsdQ) * H < ((int64_t)1 << 31);
  if (chunked) {
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SSM_ERR_LAYOUT;
    ssm_tensor_t w{};
    w.data = workspace;
    w.dtype = SSM_F32;
    w.ndim = 1;
    w.shape[0] = (int64_t)(workspace_bytes / 4);
    const ssm_tensor_t* all[] = {x, delta, A, B, C, D, dt_bias, h0, y, last_state};
    for (const ssm_tensor_t* t : all)
      if (overlaps(&w, t)) return SSM_ERR_LAYOUT;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (batch == 0) return SSM_OK;
  if (L == 0) {
    if (!last_state) return SSM_OK;
    const size_t bytes = (size_t)numel(last_state) * 4;
    const cudaError_t e = h0 ? cudaMemcpyAsync(last_state->data, h0->data, bytes, cudaMemcpyDeviceToDevice, st)
                             : cudaMemsetAsync(last_state->data, 0, bytes, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
  }
  ssm::SsdParams p;
  p.x = static_cast<const __nv_bfloat16*>(x->data);
  p.delta = static_cast<const __nv_bfloat16*>(delta->data);
  p.A = static_cast<const float*>(A->data);
  p.B = static_cast<const __nv_bfloat16*>(B->data);
  p.C = static_cast<const __nv_bfloat16*>(C->data);
  p.Dskip = D ? static_cast<const float*>(D->data) : nullptr;
  p.dt_bias = dt_bias ? static_cast<const float*>(dt_bias->data) : nullptr;
  p.dt_softplus = dt_softplus;
  p.h0 = h0 ? static_cast<const float*>(h0->data) : nullptr;
  p.y = y->data;
  p.last_state = last_state ? static_cast<float*>(last_state->data) : nullptr;
  p.batch = batch;
  p.L = L;
  p.H = H;
  p.G = groups;
  const bool yf = y->dtype == SSM_F32;
  p.nc = (int)((L + ssm::kSsdQ - 1) / ssm::kSsdQ);
  p.wait_cycles = wait_limit_cycles();
  p.fault_skip_loads = fault_skip_loads();
  p.ws_H = nullptr;
  p.ws_dt = nullptr;
  p.ws_cs = nullptr;
  p.ws_CB = nullptr;
  if (chunked) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    p.ws_H = reinterpret_cast<__nv_bfloat16*>(ws + plan.off_H);
    p.ws_dt = reinterpret_cast<float*>(ws + plan.off_dt);
    p.ws_cs = reinterpret_cast<float*>(ws + plan.off_cs);
    p.ws_CB = reinterpret_cast<float*>(ws + plan.off_CB);
  }
  cudaError_t e;
  if (P == 64 && N == 64)
    e = chunked ? launch_ssd_chunked<64, 64>(p, yf, st) : launch_ssd<64, 64>(p, yf, st);
  else if (P == 64)
    e = chunked ? launch_ssd_chunked<64, 128>(p, yf, st) : launch_ssd<64, 128>(p, yf, st);
  else if (N == 64)
    e = chunked ? launch_ssd_chunked<128, 64>(p, yf, st) : launch_ssd<128, 64>(p, yf, st);
  else
    e = chunked ? launch_ssd_chunked<128, 128>(p, yf, st) : launch_ssd<128, 128>(p, yf, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status_t ssm_device_error(void* stream, int32_t* code) {
  if (!code) return SSM_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSM_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, ssm::g_ssm_error, sizeof(int)) != cudaSuccess) return SSM_ERR_CUDA;
  if (cudaMemcpyToSymbol(ssm::g_ssm_error, &zero, sizeof(int)) != cudaSuccess) return SSM_ERR_CUDA;
  *code = v;
  return SSM_OK;
}

}  // extern "C"

// ---- forward pass with built-in scratch (allocates nothing) ---------------------------
// For callers that cannot hand the library a workspace: the segmented schedule's scratch
// (segment end states, decay products and start states) lives in this fixed array
// instead. Every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch on the current device, looked up once per device
// (with that device current) and cached; nullptr if the lookup fails.
void* noalloc_scratch() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

ssm_status_t ssm_selective_scan_fwd_noalloc(const ssm_tensor_t* u, const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                            const ssm_tensor_t* B, const ssm_tensor_t* C, const ssm_tensor_t* D,
                                            const ssm_tensor_t* z, const ssm_tensor_t* delta_bias, int delta_softplus,
                                            ssm_tensor_t* y, ssm_tensor_t* last_state, void* stream) {
  if (!u || !A) return SSM_ERR_NULL;
  if (u->ndim != 3 || A->ndim != 2) return SSM_ERR_SHAPE;
  const int64_t batch = u->shape[0], L = u->shape[1], Dm = u->shape[2], N = A->shape[1];
  if (batch < 0 || L < 0 || Dm < 0 || N < 0) return SSM_ERR_SHAPE;
  size_t need = 0;
  if (batch > 0 && L > 0 && Dm > 0 && n_supported(N)) need = plan_segments(batch, L, Dm, N).bytes;
  if (need > (size_t)SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = noalloc_scratch();
    if (!scratch) return SSM_ERR_CUDA;
  }
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, 0u, y, last_state, scratch,
                  scratch ? (size_t)SSM_NOALLOC_SCRATCH_BYTES : 0, stream);
}

}  // extern "C"
