// noalloc.cu — hla_prefill_noalloc: the prefill for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a plugin inside an engine that
// owns every byte of device memory through its own pool, a serving loop that
// may not allocate once it is running (an allocation can synchronize the
// device or fail under fragmentation at the worst moment), or a certified
// deployment that forbids allocation after start-up.  hla_prefill needs a
// caller-provided workspace for its per-segment states; this variant uses a
// fixed scratch array that lives in the library's own device memory instead,
// so the caller passes only inputs and outputs.
//
// The scratch is one file-scope __device__ array of HLA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device asks the runtime for that device's address of the array
// (cudaGetSymbolAddress, with the device current) and caches it.
//
// Under CUDA's lazy module loading (the default) the runtime loads this file's
// module, and commits the array's device memory, at that first lookup, and
// loads each kernel's module the first time the kernel is touched.  So the
// first call on a device does make the runtime commit device memory (the
// array plus the code of the kernels it runs).  An empty call (B == 0 or
// T == 0) does exactly that set-up and launches nothing: make it once per
// device at start-up, before a memory pool claims the device, and before any
// stream capture.  Calls after it allocate nothing.  (With
// CUDA_MODULE_LOADING=EAGER everything is committed when the library loads.)
// The cached address belongs to the device's current context: a process that
// destroys it (cudaDeviceReset) must not call this entry point again.
#include <mutex>

#include "hla_internal.cuh"

namespace hla {

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).  Returns HLA_ERR_CUDA if the runtime refuses.
hla_status scratch_for_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return HLA_OK;
}

// The segment plan of hla_prefill, with fewer (longer) segments when the
// per-segment states would not fit in the scratch array.
hla_status capped_plan(const hla_shape &s, Plan *out) {
  Plan p = make_plan(s);
  const size_t per_seg = (size_t)s.B * s.H * (size_t)s.dk * s.dv * sizeof(float);
  const size_t max_nseg = HLA_NOALLOC_SCRATCH_BYTES / per_seg;
  if (max_nseg < 1) return HLA_ERR_WORKSPACE;
  if ((size_t)p.nseg > max_nseg) {
    const int chunks_per_seg = ceil_div(p.nchunk, (long long)max_nseg);
    p.nseg = ceil_div(p.nchunk, chunks_per_seg);
    p.seg_len = chunks_per_seg * s.chunk;
  }
  *out = p;
  return HLA_OK;
}

}  // namespace

}  // namespace hla

using namespace hla;

extern "C" hla_status hla_prefill_noalloc(const hla_shape *s, const void *q, const void *k,
                                          const void *v, const void *gate, const float *gamma,
                                          const float *state_in, float *state_out, void *y,
                                          float *o, hla_stream stream) {
  hla_status st = check_shape(s, false);
  if (st != HLA_OK) return st;
  if ((st = check_gamma(gamma, s->H)) != HLA_OK) return st;
  const bool empty = s->B == 0 || s->T == 0;
  const void *required[] = {q, k, v, gate, y};
  for (const void *p : required)
    if ((st = need_unless(empty, p)) != HLA_OK) return st;
  const void *optional[] = {state_in, state_out, o};
  for (const void *p : optional)
    if ((st = maybe(p)) != HLA_OK) return st;
  Plan plan;
  if (!empty && (st = capped_plan(*s, &plan)) != HLA_OK) return st;
  // per-device set-up: the scratch array's address, and the kernels this
  // shape runs loaded (an empty call does only this)
  void *scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != HLA_OK) return st;
  if (prepare_simt_forward(s->dtype, s->dk) != cudaSuccess || prepare_state_scan() != cudaSuccess)
    return HLA_ERR_CUDA;
  if (empty)
    return pass_state(*s, state_in, state_out, (cudaStream_t)stream) == cudaSuccess ? HLA_OK
                                                                                   : HLA_ERR_CUDA;

  MixerParams P;
  fill_common(P, *s, gamma);
  P.nseg = plan.nseg;
  P.seg_len = plan.seg_len;
  P.q = q;
  P.k = k;
  P.v = v;
  P.g = gate;
  P.state_in = state_in;
  P.state_out = state_out;
  P.y = y;
  P.o = o;
  P.seg = (float *)scratch;  // fully written by the first pass: nothing to clear
  cudaStream_t cs = (cudaStream_t)stream;
  if (launch_simt_seg_state(P, s->dtype, cs) != cudaSuccess) return HLA_ERR_CUDA;
  if (launch_state_scan(P, state_out != nullptr, cs) != cudaSuccess) return HLA_ERR_CUDA;
  if (launch_simt_seg_output(P, s->dtype, cs) != cudaSuccess) return HLA_ERR_CUDA;
  return HLA_OK;
}
