// C ABI of libselscan: host-side argument checks, then one kernel launch on the caller's stream.
// Nothing is enqueued unless every check passes.  See include/selscan.h for the contract.
#include <cudaTypedefs.h>

#include <climits>
#include <cstdlib>
#include <cstring>
#include <cstdint>
#include <mutex>

#include "selscan_internal.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

selscan_status_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return SELSCAN_ERR_CUDA;
}

// cuMemGetAddressRange, fetched through the runtime so the library does not link libcuda.
PFN_cuMemGetAddressRange_v3020 g_get_range = nullptr;
void* g_encode_tiled = nullptr;
std::once_flag g_range_once;

void init_range_query() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_get_range = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode_tiled = fn;
}

bool mul_ok(int64_t a, int64_t b, int64_t* r) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *r = a * b;
  return true;
}

size_t dsize(selscan_dtype_t t) { return t == SELSCAN_BF16 ? 2 : 4; }

// One tensor argument: its address and byte extent.
struct Span {
  const void* p;
  int64_t bytes;
};

// The pointer must be device-accessible; for device and managed memory its whole extent must lie
// inside the allocation that contains it (pinned host memory is accepted without an extent check).
selscan_status_t check_pointer(const Span& s) {
  if (s.bytes == 0) return SELSCAN_OK;
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, s.p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error so later calls are unaffected
    return SELSCAN_ERR_POINTER;
  }
  if (attr.type == cudaMemoryTypeUnregistered) return SELSCAN_ERR_POINTER;
  if (attr.type == cudaMemoryTypeHost) return attr.devicePointer ? SELSCAN_OK : SELSCAN_ERR_POINTER;
  if (attr.type == cudaMemoryTypeDevice) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != attr.device) return SELSCAN_ERR_POINTER;
  }
  std::call_once(g_range_once, init_range_query);
  if (!g_get_range) return SELSCAN_ERR_POINTER;  // the extent cannot be checked: refuse rather than risk a fault
  CUdeviceptr base = 0;
  size_t size = 0;
  if (g_get_range(&base, &size, reinterpret_cast<CUdeviceptr>(s.p)) != CUDA_SUCCESS) return SELSCAN_ERR_POINTER;
  const uintptr_t p = reinterpret_cast<uintptr_t>(s.p);
  if (p < base || p - base > size || static_cast<uint64_t>(s.bytes) > size - (p - base)) return SELSCAN_ERR_POINTER;
  return SELSCAN_OK;
}

bool overlaps(const Span& a, const Span& b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + static_cast<uint64_t>(b.bytes) && b0 < a0 + static_cast<uint64_t>(a.bytes);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

selscan_status_t check_shape(const selscan_shape_t* s) {
  if (!s) return SELSCAN_ERR_NULL;
  if (s->batch < 0 || s->dim < 0 || s->seqlen < 0 || s->dstate < 1) return SELSCAN_ERR_SHAPE;
  if (s->in_dtype != SELSCAN_F32 && s->in_dtype != SELSCAN_BF16) return SELSCAN_ERR_UNSUPPORTED;
  if (s->out_dtype != SELSCAN_F32 && s->out_dtype != SELSCAN_BF16) return SELSCAN_ERR_UNSUPPORTED;
  if (s->dstate > SELSCAN_MAX_DSTATE) return SELSCAN_ERR_UNSUPPORTED;
  return SELSCAN_OK;
}

// Shared checks of the argument lists: sizes, nulls, alignment, device extents, aliasing.
// `outs` are written by the call; an output may coincide exactly with the input named `may_alias`.
selscan_status_t check_args(const Span* ins, const bool* required_in, const size_t* elem_in, int n_in,
                            const Span* outs, const bool* required_out, const size_t* elem_out, int n_out,
                            const void* may_alias_in, const void* may_alias_out) {
  for (int i = 0; i < n_in; i++)
    if (required_in[i] && !ins[i].p && ins[i].bytes > 0) return SELSCAN_ERR_NULL;
  for (int i = 0; i < n_out; i++)
    if (required_out[i] && !outs[i].p && outs[i].bytes > 0) return SELSCAN_ERR_NULL;
  for (int i = 0; i < n_in; i++)
    if (ins[i].p && !aligned(ins[i].p, elem_in[i])) return SELSCAN_ERR_ALIGN;
  for (int i = 0; i < n_out; i++)
    if (outs[i].p && !aligned(outs[i].p, elem_out[i])) return SELSCAN_ERR_ALIGN;
  for (int i = 0; i < n_in; i++)
    if (ins[i].p) {
      selscan_status_t st = check_pointer(ins[i]);
      if (st != SELSCAN_OK) return st;
    }
  for (int i = 0; i < n_out; i++)
    if (outs[i].p) {
      selscan_status_t st = check_pointer(outs[i]);
      if (st != SELSCAN_OK) return st;
    }
  for (int o = 0; o < n_out; o++) {
    for (int i = 0; i < n_in; i++) {
      if (!overlaps(outs[o], ins[i])) continue;
      const bool allowed = may_alias_out && outs[o].p == may_alias_out && ins[i].p == may_alias_in &&
                           outs[o].bytes == ins[i].bytes;
      if (!allowed) return SELSCAN_ERR_ALIAS;
    }
    for (int o2 = o + 1; o2 < n_out; o2++)
      if (overlaps(outs[o], outs[o2])) return SELSCAN_ERR_ALIAS;
  }
  return SELSCAN_OK;
}

}  // namespace

namespace selscan {
thread_local int t_launches = 0;
void count_launches(int n) { t_launches += n; }
void* tensor_map_encoder() {
  std::call_once(g_range_once, init_range_query);
  return g_encode_tiled;
}
}  // namespace selscan

namespace {

// The checks shared by every forward entry point, and the launch arguments they produce.  *done is set
// when nothing is left to launch: no rows, or an empty sequence (h_last = h0 or zeros, written here
// by a copy or a fill, which allocate nothing).
selscan_status_t prepare_fwd(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                             const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                             int delta_softplus, const float* h0, void* out, float* h_last, bool conv,
                             const float* conv_w, const float* conv_b, cudaStream_t s, selscan::FwdParams* p,
                             bool* done, float* ckpt = nullptr) {
  *done = false;
  selscan::t_launches = 0;
  if (conv && !conv_w) return SELSCAN_ERR_NULL;
  selscan_status_t st = check_shape(shape);
  if (st != SELSCAN_OK) return st;
  const int64_t Bsz = shape->batch, Dm = shape->dim, L = shape->seqlen, N = shape->dstate;
  int64_t rows, elems, bcn, bc_elems, an, states;
  if (!mul_ok(Bsz, Dm, &rows) || !mul_ok(rows, L, &elems) || !mul_ok(Bsz, N, &bcn) || !mul_ok(bcn, L, &bc_elems) ||
      !mul_ok(Dm, N, &an) || !mul_ok(rows, N, &states))
    return SELSCAN_ERR_SHAPE;
  if (elems > INT64_MAX / 4 || bc_elems > INT64_MAX / 4 || states > INT64_MAX / 4) return SELSCAN_ERR_SHAPE;
  if (Bsz > 65535) return SELSCAN_ERR_UNSUPPORTED;  // one grid row per batch entry
  const size_t ei = dsize(shape->in_dtype), eo = dsize(shape->out_dtype);
  const Span ins[] = {{u, elems * (int64_t)ei},     {delta, elems * (int64_t)ei}, {A, an * 4},
                      {B, bc_elems * (int64_t)ei},  {C, bc_elems * (int64_t)ei},  {D, Dm * 4},
                      {z, elems * (int64_t)ei},     {delta_bias, Dm * 4},         {h0, states * 4},
                      {conv ? conv_w : nullptr, Dm * 16}, {conv ? conv_b : nullptr, Dm * 4}};
  const bool req_in[] = {true, true, true, true, true, false, false, false, false, conv, false};
  const size_t el_in[] = {ei, ei, 4, ei, ei, 4, ei, 4, 4, 4, 4};
  const int64_t nck = (L + 15) / 16;  // 16-step checkpoint chunks
  int64_t ck_floats;
  if (!mul_ok(rows, nck * 16, &ck_floats) || ck_floats > INT64_MAX / 4) return SELSCAN_ERR_SHAPE;
  const Span outs[] = {{out, elems * (int64_t)eo}, {h_last, states * 4}, {ckpt, ck_floats * 4}};
  const bool req_out[] = {true, false, false};
  const size_t el_out[] = {eo, 4, 16};
  st = check_args(ins, req_in, el_in, 11, outs, req_out, el_out, 3, h0, h_last);
  if (st != SELSCAN_OK) return st;
  if (rows == 0) {
    *done = true;
    return SELSCAN_OK;
  }
  if (L == 0) {  // empty sequence: the state passes through unchanged
    *done = true;
    if (h_last && h_last != h0) {
      cudaError_t e = h0 ? cudaMemcpyAsync(h_last, h0, states * 4, cudaMemcpyDeviceToDevice, s)
                         : cudaMemsetAsync(h_last, 0, states * 4, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return SELSCAN_OK;
  }
  memset(p, 0, sizeof *p);
  p->batch = Bsz;
  p->dim = Dm;
  p->seqlen = L;
  p->dstate = static_cast<int>(N);
  p->u = u;
  p->delta = delta;
  p->z = z;
  p->B = B;
  p->C = C;
  p->A = A;
  p->D = D;
  p->delta_bias = delta_bias;
  p->h0 = h0;
  p->out = out;
  p->h_last = h_last;
  p->delta_softplus = delta_softplus != 0;
  const int64_t vin = 16 / ei, vout = 16 / eo;
  p->vec_in = aligned(u, 16) && aligned(delta, 16) && (!z || aligned(z, 16)) && L % vin == 0;
  p->vec_out = aligned(out, 16) && L % vout == 0;
  p->vec_bc = aligned(B, 16) && aligned(C, 16) && L % vin == 0;
  p->vec_stage = p->vec_bc && p->vec_in;  // u, delta, z rows may be bulk-copied too
  p->tblock = L;
  p->nblocks = 1;
  p->conv_w = conv ? conv_w : nullptr;
  p->conv_b = conv ? conv_b : nullptr;
  p->out_bf16 = shape->out_dtype == SELSCAN_BF16;
  p->ckpt = ckpt;
  p->ckpt_chunks = nck;
  return SELSCAN_OK;
}

// The row-sequential kernel unless it cannot stage the inputs or SELSCAN_KERNEL forces an older one.
bool rows_path(const selscan::FwdParams& p, selscan_dtype_t in_dtype) {
  const char* k = getenv("SELSCAN_KERNEL");
  return (!k || k[0] == 'r') && selscan::rows_kernel_supports(p, in_dtype);
}

}  // namespace

extern "C" {

selscan_status_t selscan_fwd(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* delta_bias, int delta_softplus, const float* h0, void* out,
                             float* h_last, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selscan::FwdParams p;
  bool done = false;
  selscan_status_t st = prepare_fwd(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out, h_last,
                                    false, nullptr, nullptr, s, &p, &done);
  if (st != SELSCAN_OK || done) return st;
  cudaError_t e = selscan::launch_fwd(p, shape->in_dtype, shape->out_dtype, s);
  return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e);
}

// selscan_fwd with the reverse direction and/or the exact zero-order-hold input matrix.
selscan_status_t selscan_fwd_ex(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                const void* B, const void* C, const float* D, const void* z,
                                const float* delta_bias, int delta_softplus, const float* h0, void* out,
                                float* h_last, unsigned flags, void* stream) {
  if (flags & ~(SELSCAN_FLAG_REVERSE | SELSCAN_FLAG_ZOH)) return SELSCAN_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selscan::FwdParams p;
  bool done = false;
  selscan_status_t st = prepare_fwd(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out, h_last,
                                    false, nullptr, nullptr, s, &p, &done);
  if (st != SELSCAN_OK || done) return st;
  const bool rev = (flags & SELSCAN_FLAG_REVERSE) != 0, zoh = (flags & SELSCAN_FLAG_ZOH) != 0;
  cudaError_t e;
  if (rows_path(p, shape->in_dtype)) {
    selscan::RowsOptions o;
    o.reverse = rev;
    o.zoh = zoh;
    e = selscan::launch_fwd_rows(p, shape->in_dtype, shape->out_dtype, o, s, nullptr);
  } else {
    e = selscan::launch_fwd_seq_ex(p, shape->in_dtype, shape->out_dtype, rev, zoh, s);
  }
  return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e);
}

// The forward with the block's convolution front: u = silu(conv_b + causal depthwise conv1d(x, conv_w)),
// computed in the kernel from x (passed where selscan_fwd takes u).  The checks of selscan_fwd, plus
// conv_w [D, 4] fp32 (required) and conv_b [D] fp32 (optional).
selscan_status_t selscan_fwd_conv(const selscan_shape_t* shape, const void* u, const float* conv_w,
                                  const float* conv_b, const void* delta, const float* A, const void* B,
                                  const void* C, const float* D, const void* z, const float* delta_bias,
                                  int delta_softplus, const float* h0, void* out, float* h_last, unsigned flags,
                                  void* stream) {
  if (flags & ~SELSCAN_FLAG_ZOH) return SELSCAN_ERR_UNSUPPORTED;  // the front is causal: no reverse
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selscan::FwdParams p;
  bool done = false;
  selscan_status_t st = prepare_fwd(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out, h_last,
                                    true, conv_w, conv_b, s, &p, &done);
  if (st != SELSCAN_OK || done) return st;
  const bool zoh = (flags & SELSCAN_FLAG_ZOH) != 0;
  cudaError_t e;
  if (rows_path(p, shape->in_dtype)) {
    selscan::RowsOptions o;
    o.zoh = zoh;
    o.conv = true;
    e = selscan::launch_fwd_rows(p, shape->in_dtype, shape->out_dtype, o, s, nullptr);
  } else {
    e = selscan::launch_fwd_seq_ex(p, shape->in_dtype, shape->out_dtype, false, zoh, s, true);
  }
  return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e);
}

// For callers that may not allocate device memory while they run: the checks of selscan_fwd, then the
// forward with its time-block scratch in the library's fixed device array.
selscan_status_t selscan_fwd_noalloc(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                     const void* B, const void* C, const float* D, const void* z,
                                     const float* delta_bias, int delta_softplus, const float* h0, void* out,
                                     float* h_last, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selscan::FwdParams p;
  bool done = false;
  selscan_status_t st = prepare_fwd(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out, h_last,
                                    false, nullptr, nullptr, s, &p, &done);
  if (st != SELSCAN_OK || done) return st;
  bool too_big = false;
  cudaError_t e;
  if (rows_path(p, shape->in_dtype)) {
    selscan::RowsOptions o;
    o.scratch = selscan::ScratchSource::Fixed;
    e = selscan::launch_fwd_rows(p, shape->in_dtype, shape->out_dtype, o, s, &too_big);
  } else {
    e = selscan::launch_fwd_seq_noalloc(p, shape->in_dtype, shape->out_dtype, s, &too_big);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return too_big ? SELSCAN_ERR_SCRATCH : SELSCAN_OK;
}

size_t selscan_bwd_workspace_size(const selscan_shape_t* shape) {
  if (check_shape(shape) != SELSCAN_OK) return 0;
  int64_t rows, elems;
  if (!mul_ok(shape->batch, shape->dim, &rows) || !mul_ok(rows, shape->seqlen, &elems) || elems > INT64_MAX / 16)
    return 0;
  return selscan::bwd_workspace_bytes(shape->batch, shape->dim, shape->seqlen);
}

}  // extern "C"

namespace {

// The backward: the checks of the forward's inputs plus dout, dh_last, the checkpoints (optional) and the
// gradient outputs, zeroing of the accumulated gradients, then its kernels.
selscan_status_t bwd_impl(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                          const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                          int delta_softplus, const float* h0, const void* dout, const float* dh_last,
                          const float* ckpt, void* du, void* ddelta, void* dz, float* dA, float* dB, float* dC,
                          float* dD, float* ddelta_bias, float* dh0, void* workspace, size_t workspace_bytes,
                          void* stream) {
  selscan::t_launches = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selscan_status_t st = check_shape(shape);
  if (st != SELSCAN_OK) return st;
  if (z && !dz) return SELSCAN_ERR_NULL;
  if (!z) dz = nullptr;
  const int64_t Bsz = shape->batch, Dm = shape->dim, L = shape->seqlen, N = shape->dstate;
  int64_t rows, elems, bcn, bc_elems, an, states;
  if (!mul_ok(Bsz, Dm, &rows) || !mul_ok(rows, L, &elems) || !mul_ok(Bsz, N, &bcn) || !mul_ok(bcn, L, &bc_elems) ||
      !mul_ok(Dm, N, &an) || !mul_ok(rows, N, &states))
    return SELSCAN_ERR_SHAPE;
  if (elems > INT64_MAX / 16 || bc_elems > INT64_MAX / 4 || states > INT64_MAX / 4) return SELSCAN_ERR_SHAPE;
  if (Bsz > 65535) return SELSCAN_ERR_UNSUPPORTED;  // one grid row per batch entry
  const size_t ei = dsize(shape->in_dtype), eo = dsize(shape->out_dtype);
  const size_t ws_need = selscan::bwd_workspace_bytes(Bsz, Dm, L, ckpt == nullptr);
  if (workspace && workspace_bytes < ws_need) return SELSCAN_ERR_SCRATCH;
  const int64_t ck_floats = rows * ((L + 15) / 16) * 16;
  const Span ins[] = {{u, elems * (int64_t)ei},    {delta, elems * (int64_t)ei}, {A, an * 4},
                      {B, bc_elems * (int64_t)ei}, {C, bc_elems * (int64_t)ei},  {D, Dm * 4},
                      {z, elems * (int64_t)ei},    {delta_bias, Dm * 4},         {h0, states * 4},
                      {dout, elems * (int64_t)eo}, {dh_last, states * 4},        {ckpt, ck_floats * 4}};
  const bool req_in[] = {true, true, true, true, true, false, false, false, false, true, false, false};
  const size_t el_in[] = {ei, ei, 4, ei, ei, 4, ei, 4, 4, eo, 4, 16};
  const Span outs[] = {{du, elems * (int64_t)ei}, {ddelta, elems * (int64_t)ei}, {dz, elems * (int64_t)ei},
                       {dA, an * 4},              {dB, bc_elems * 4},             {dC, bc_elems * 4},
                       {dD, Dm * 4},              {ddelta_bias, Dm * 4},          {dh0, states * 4},
                       {workspace, (int64_t)ws_need}};
  const bool req_out[] = {true, true, false, true, true, true, false, false, false, false};
  const size_t el_out[] = {ei, ei, ei, 4, 4, 4, 4, 4, 4, 16};
  st = check_args(ins, req_in, el_in, 12, outs, req_out, el_out, 10, nullptr, nullptr);
  if (st != SELSCAN_OK) return st;
  // The accumulated gradients start from zero (stream-ordered fills, no allocation).
  cudaError_t e = cudaSuccess;
  const struct {
    void* p;
    int64_t bytes;
  } zero[] = {{dA, an * 4}, {dB, bc_elems * 4}, {dC, bc_elems * 4}, {dD, Dm * 4}, {ddelta_bias, Dm * 4}};
  for (const auto& zf : zero)
    if (zf.p && zf.bytes > 0 && e == cudaSuccess) e = cudaMemsetAsync(zf.p, 0, zf.bytes, s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (rows == 0) return SELSCAN_OK;
  if (L == 0) {  // no steps: the state's gradient passes through unchanged
    if (dh0) {
      e = dh_last ? cudaMemcpyAsync(dh0, dh_last, states * 4, cudaMemcpyDeviceToDevice, s)
                  : cudaMemsetAsync(dh0, 0, states * 4, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return SELSCAN_OK;
  }
  selscan::BwdParams p;
  memset(&p, 0, sizeof p);
  p.batch = Bsz;
  p.dim = Dm;
  p.seqlen = L;
  p.dstate = static_cast<int>(N);
  p.u = u;
  p.delta = delta;
  p.z = z;
  p.B = B;
  p.C = C;
  p.A = A;
  p.D = D;
  p.delta_bias = delta_bias;
  p.h0 = h0;
  p.dout = dout;
  p.dh_last = dh_last;
  p.du = du;
  p.ddelta = ddelta;
  p.dz = dz;
  p.dA = dA;
  p.dB = dB;
  p.dC = dC;
  p.dD = dD;
  p.ddelta_bias = ddelta_bias;
  p.dh0 = dh0;
  p.ckpt_in = ckpt;
  p.delta_softplus = delta_softplus != 0;
  p.vec_in = aligned(u, 4 * ei) && aligned(delta, 4 * ei) && (!z || aligned(z, 4 * ei)) && L % 4 == 0;
  p.vec_dout = aligned(dout, 4 * eo) && L % 4 == 0;
  p.vec_grad = aligned(du, 4 * ei) && aligned(ddelta, 4 * ei) && (!dz || aligned(dz, 4 * ei)) && L % 4 == 0;
  p.vec_dbc = aligned(dB, 16) && aligned(dC, 16) && L % 4 == 0;
  e = selscan::launch_bwd(p, shape->in_dtype, shape->out_dtype, workspace, s);
  return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

selscan_status_t selscan_bwd(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* delta_bias, int delta_softplus, const float* h0, const void* dout,
                             const float* dh_last, void* du, void* ddelta, void* dz, float* dA, float* dB,
                             float* dC, float* dD, float* ddelta_bias, float* dh0, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return bwd_impl(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, dout, dh_last, nullptr, du, ddelta,
                  dz, dA, dB, dC, dD, ddelta_bias, dh0, workspace, workspace_bytes, stream);
}

// selscan_bwd from the checkpoints selscan_fwd_ckpt kept (the backward's own forward pass is skipped).
selscan_status_t selscan_bwd_ckpt(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus, const float* h0, const void* dout,
                                  const float* dh_last, const float* ckpt, void* du, void* ddelta, void* dz,
                                  float* dA, float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!ckpt && shape && shape->batch > 0 && shape->dim > 0 && shape->seqlen > 0) return SELSCAN_ERR_NULL;
  return bwd_impl(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, dout, dh_last, ckpt, du, ddelta,
                  dz, dA, dB, dC, dD, ddelta_bias, dh0, workspace, workspace_bytes, stream);
}

// The forward that also keeps the state before every 16-step chunk for the backward (selscan_bwd_ckpt).
selscan_status_t selscan_fwd_ckpt(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus, const float* h0, void* out,
                                  float* h_last, float* ckpt, void* stream) {
  if (!ckpt && shape && shape->batch > 0 && shape->dim > 0 && shape->seqlen > 0) return SELSCAN_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selscan::FwdParams p;
  bool done = false;
  selscan_status_t st = prepare_fwd(shape, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out, h_last,
                                    false, nullptr, nullptr, s, &p, &done, ckpt);
  if (st != SELSCAN_OK || done) return st;
  if (!selscan::rows_kernel_supports(p, shape->in_dtype)) return SELSCAN_ERR_UNSUPPORTED;
  const cudaError_t e = selscan::launch_fwd_rows(p, shape->in_dtype, shape->out_dtype, selscan::RowsOptions{}, s,
                                                 nullptr);
  return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e);
}

selscan_status_t selscan_step(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              const float* delta_bias, int delta_softplus, float* state, void* out,
                              void* stream) {
  selscan::t_launches = 0;
  selscan_status_t st = check_shape(shape);
  if (st != SELSCAN_OK) return st;
  if (shape->seqlen != 1) return SELSCAN_ERR_SHAPE;
  const int64_t Bsz = shape->batch, Dm = shape->dim, N = shape->dstate;
  int64_t rows, bcn, an, states;
  if (!mul_ok(Bsz, Dm, &rows) || !mul_ok(Bsz, N, &bcn) || !mul_ok(Dm, N, &an) || !mul_ok(rows, N, &states))
    return SELSCAN_ERR_SHAPE;
  if (states > INT64_MAX / 4 || rows > (int64_t)INT32_MAX * 64) return SELSCAN_ERR_SHAPE;
  const size_t ei = dsize(shape->in_dtype), eo = dsize(shape->out_dtype);
  const Span ins[] = {{u, rows * (int64_t)ei}, {delta, rows * (int64_t)ei}, {A, an * 4},
                      {B, bcn * (int64_t)ei},  {C, bcn * (int64_t)ei},      {D, Dm * 4},
                      {z, rows * (int64_t)ei}, {delta_bias, Dm * 4}};
  const bool req_in[] = {true, true, true, true, true, false, false, false};
  const size_t el_in[] = {ei, ei, 4, ei, ei, 4, ei, 4};
  const Span outs[] = {{state, states * 4}, {out, rows * (int64_t)eo}};
  const bool req_out[] = {true, true};
  const size_t el_out[] = {4, eo};
  st = check_args(ins, req_in, el_in, 8, outs, req_out, el_out, 2, nullptr, nullptr);
  if (st != SELSCAN_OK) return st;
  if (rows == 0) return SELSCAN_OK;
  selscan::StepParams p;
  p.batch = Bsz;
  p.dim = Dm;
  p.dstate = static_cast<int>(N);
  p.u = u;
  p.delta = delta;
  p.z = z;
  p.B = B;
  p.C = C;
  p.A = A;
  p.D = D;
  p.delta_bias = delta_bias;
  p.state = state;
  p.out = out;
  p.delta_softplus = delta_softplus != 0;
  p.vec_state = (N % 4 == 0) && aligned(state, 16) && aligned(A, 16);
  p.vec_bc = aligned(B, 4 * ei) && aligned(C, 4 * ei);
  cudaError_t e = selscan::launch_step(p, shape->in_dtype, shape->out_dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e);
}

const char* selscan_status_string(selscan_status_t status) {
  switch (status) {
    case SELSCAN_OK: return "SELSCAN_OK";
    case SELSCAN_ERR_NULL: return "SELSCAN_ERR_NULL: a required pointer is NULL";
    case SELSCAN_ERR_SHAPE: return "SELSCAN_ERR_SHAPE: invalid or overflowing sizes";
    case SELSCAN_ERR_ALIGN: return "SELSCAN_ERR_ALIGN: a pointer is not aligned to its element size";
    case SELSCAN_ERR_UNSUPPORTED: return "SELSCAN_ERR_UNSUPPORTED: dstate or dtype not supported";
    case SELSCAN_ERR_CUDA: return "SELSCAN_ERR_CUDA: a CUDA call failed";
    case SELSCAN_ERR_POINTER: return "SELSCAN_ERR_POINTER: pointer not device-accessible or extent outside its allocation";
    case SELSCAN_ERR_ALIAS: return "SELSCAN_ERR_ALIAS: an output overlaps an input";
    case SELSCAN_ERR_SCRATCH:
      return "SELSCAN_ERR_SCRATCH: the problem needs more scratch than the buffer it may use (selscan_fwd_noalloc's "
             "fixed array, or selscan_bwd's workspace)";
  }
  return "unknown selscan status";
}

int selscan_last_cuda_error(void) { return g_last_cuda_error; }

int selscan_device_status(int reset) {
  int v = 0, w = 0;
  if (selscan::read_device_error(&v, reset) != cudaSuccess) return -1;
  if (selscan::read_seq_device_error(&w, reset) != cudaSuccess) return -1;
  int x = 0;
  if (selscan::read_rows_device_error(&x, reset) != cudaSuccess) return -1;
  return v | w | x;
}

int selscan_abi_version(void) { return SELSCAN_ABI_VERSION; }

int selscan_last_launch_count(void) { return selscan::t_launches; }

}  // extern "C"
