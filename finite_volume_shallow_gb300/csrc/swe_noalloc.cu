// swe_noalloc.cu -- swe_run_noalloc: the time loop on caller-owned device
// buffers, with every piece of scratch memory in one file-scope device array.
//
// Who needs it: callers that must not allocate device memory after start-up
// -- a framework that already owns (pre-allocates) nearly all of the GPU's
// memory through its own pool, so a cudaMalloc would fail or fragment it, and
// real-time or embedded loops that forbid allocation because cudaMalloc can
// block, synchronise the device and fragment memory.  They pass inputs and
// outputs; the scratch of the step (wave-speed maxima, error word, clock, dt
// history) lives in g_noalloc_scratch below.
//
// g_noalloc_scratch is a host-side stand-in in host code: its device address
// is obtained once per device with cudaGetSymbolAddress and passed to the
// kernels.  CUDA loads device code lazily, so the array is reserved on a
// device by the first call there (which also does that look-up) and held
// until the process exits.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/swe.h"
#include "swe_internal.h"
#include "swe_plan.h"

using namespace swe;

namespace {

// scratch layout (bytes): [0, 24) three wave-speed maxima, [64, 68) error
// word, [128, 136) simulated time, [256, 256 + 8 * max steps) dt of each step
constexpr size_t kSlotsOff = 0;
constexpr size_t kErrOff = 64;
constexpr size_t kTimeOff = 128;
constexpr size_t kDtsOff = 256;
constexpr size_t kScratchBytes = kDtsOff + 8 * (size_t)SWE_NOALLOC_MAX_STEPS;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_dev[kMaxDevices] = {nullptr};
bool g_attr_done[kMaxDevices][4] = {{false}};  // [precision + 2 * entropy fix]
int g_blocks_per_sm[kMaxDevices][4] = {{0}};
int g_sms[kMaxDevices] = {0};

swe_status cuda_st(cudaError_t e) {
  if (e == cudaSuccess) return SWE_OK;
  (void)cudaGetLastError();
  return SWE_ERR_CUDA;
}

#define CKN(call)                                  \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_st(e_);     \
  } while (0)

// Once per device (with that device current): the scratch array's device
// address, the step kernel's shared-memory attribute and its occupancy.
template <typename T>
swe_status setup(int dev, bool efix, unsigned char** scratch, int* bpsm, int* sms) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const int ti = (sizeof(T) == 4 ? 0 : 1) + (efix ? 2 : 0);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    CKN(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    g_scratch_dev[dev] = static_cast<unsigned char*>(p);
    CKN(cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev));
  }
  if (!g_attr_done[dev][ti]) {
    size_t smem = 0;
    CKN(step_occupancy<T>(&g_blocks_per_sm[dev][ti], &smem, efix));
    if (g_blocks_per_sm[dev][ti] < 1) return SWE_ERR_CUDA;
    g_attr_done[dev][ti] = true;
  }
  *scratch = g_scratch_dev[dev];
  *bpsm = g_blocks_per_sm[dev][ti];
  *sms = g_sms[dev];
  return SWE_OK;
}

template <typename T>
swe_status run(const swe_grid* g, const swe_params* p, const void* H, void* const* Wa,
               void* const* Wb, int32_t pitch, int64_t nsteps, double* dts_out) {
  int dev = 0;
  CKN(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return SWE_ERR_UNSUPPORTED;
  unsigned char* scr = nullptr;
  int bpsm = 0, sms = 0;
  swe_status st = setup<T>(dev, p->entropy_fix != 0, &scr, &bpsm, &sms);
  if (st != SWE_OK) return st;
  cudaStream_t stream = (cudaStream_t)p->stream;

  // launch shape: the same rule as a handle's (one warp per column band and
  // row segment, about one unit per resident warp, segments >= 32 rows)
  const int own = band_owned<T>();
  const int nbands = (g->nx + own - 1) / own;
  const StepPlan pl = plan_step((int64_t)sms * bpsm * kWarpsPerBlock, nbands, g->ny);
  const int blocks = (pl.units + kWarpsPerBlock - 1) / kWarpsPerBlock;

  // scratch that must start at zero: maxima, error word, clock
  CKN(cudaMemsetAsync(scr, 0, kDtsOff, stream));
  void* slots = scr + kSlotsOff;
  unsigned* err = reinterpret_cast<unsigned*>(scr + kErrOff);
  double* tdev = reinterpret_cast<double*>(scr + kTimeOff);
  double* dts = reinterpret_cast<double*>(scr + kDtsOff);

  const T* a[4] = {(const T*)Wa[0], (const T*)Wa[1], (const T*)Wa[2], (const T*)Wa[3]};
  const T gh = (T)(0.5 * p->g);
  const T rho = (T)(g->dx / g->dy);
  CKN(launch_dt0<T>(a, (const T*)H, g->nx, g->ny, pitch, gh, rho, slots, err, stream));
  for (int64_t n = 0; n < nsteps; ++n) {
    void* const* in = (n % 2 == 0) ? Wa : Wb;
    void* const* out = (n % 2 == 0) ? Wb : Wa;
    StepArgs<T> s;
    for (int f = 0; f < 4; ++f) {
      s.win[f] = (const T*)in[f];
      s.wout[f] = (T*)out[f];
    }
    s.H = (const T*)H;
    s.nx = g->nx;
    s.ny = g->ny;
    s.pitch = pitch;
    s.nbands = nbands;
    s.nsegs = pl.nsegs;
    s.nsegs_wall = pl.nsegs_wall;
    s.ghalf = gh;
    s.rho = rho;
    s.two_cfl = 2.0 * p->cfl;
    s.dx = g->dx;
    s.tmax_in = (char*)slots + (n % 3) * 8;
    s.tmax_out = (char*)slots + ((n + 1) % 3) * 8;
    s.tmax_clear = (char*)slots + ((n + 2) % 3) * 8;
    s.dt_hist = dts;
    s.t_dev = tdev;
    s.step = n;
    s.err = err;
    s.efix = p->entropy_fix;
    CKN(launch_step<T>(s, blocks, stream));
  }
  if (nsteps % 2 == 1) {  // the state is in Wb: hand it back in Wa
    const size_t bytes = (size_t)(g->ny + 2 * kPadY) * (size_t)pitch * sizeof(T);
    for (int f = 0; f < 4; ++f)
      CKN(cudaMemcpyAsync(Wa[f], Wb[f], bytes, cudaMemcpyDeviceToDevice, stream));
  }
  unsigned bits = 0;
  CKN(cudaMemcpyAsync(&bits, err, sizeof(unsigned), cudaMemcpyDeviceToHost, stream));
  if (dts_out && nsteps > 0)
    CKN(cudaMemcpyAsync(dts_out, dts, (size_t)nsteps * sizeof(double), cudaMemcpyDeviceToHost,
                        stream));
  CKN(cudaStreamSynchronize(stream));
  if (bits & kErrTimeout) return SWE_ERR_TIMEOUT;
  if (bits & kErrNonfinite) return SWE_ERR_NONFINITE;
  if (bits & kErrDepth) return SWE_ERR_DEPTH;
  return SWE_OK;
}

bool pos_finite(double v) { return isfinite(v) && v > 0.0; }

}  // namespace

extern "C" swe_status swe_run_noalloc(const swe_grid* grid, const swe_params* params,
                                      const void* H, void* const* W_a, void* const* W_b,
                                      int32_t pitch, int64_t nsteps, double* dts_out) {
  if (!grid || !params || !H || !W_a || !W_b) return SWE_ERR_ARG;
  for (int f = 0; f < 4; ++f)
    if (!W_a[f] || !W_b[f]) return SWE_ERR_ARG;
  if (grid->nx < 1 || grid->ny < 1 || grid->nx > (1 << 30) || grid->ny > (1 << 30) - 8)
    return SWE_ERR_ARG;
  if (!pos_finite(grid->dx) || !pos_finite(grid->dy)) return SWE_ERR_ARG;
  if (params->precision != 32 && params->precision != 64) return SWE_ERR_ARG;
  if (!pos_finite(params->g) || !(params->cfl > 0.0 && params->cfl <= 1.0)) return SWE_ERR_ARG;
  if (params->n_layers == 2 || params->pollutant != 1) return SWE_ERR_UNSUPPORTED;
  if (params->wet_dry != 0) return SWE_ERR_UNSUPPORTED;
  if (params->entropy_fix != 0 && params->entropy_fix != 1) return SWE_ERR_ARG;
  if (params->n_layers != 1) return SWE_ERR_ARG;
  if (nsteps < 0 || nsteps > SWE_NOALLOC_MAX_STEPS) return SWE_ERR_ARG;
  const int64_t need =
      params->precision == 32 ? grid_pitch<float>(grid->nx) : grid_pitch<double>(grid->nx);
  if (pitch < need || pitch % 32 != 0) return SWE_ERR_ARG;
  const uintptr_t align = 16;
  if ((uintptr_t)H % align) return SWE_ERR_ARG;
  for (int f = 0; f < 4; ++f)
    if ((uintptr_t)W_a[f] % align || (uintptr_t)W_b[f] % align) return SWE_ERR_ARG;
  return params->precision == 32
             ? run<float>(grid, params, H, W_a, W_b, pitch, nsteps, dts_out)
             : run<double>(grid, params, H, W_a, W_b, pitch, nsteps, dts_out);
}
