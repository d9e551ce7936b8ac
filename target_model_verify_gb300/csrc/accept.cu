// Acceptance test and first-reject scan, one CTA per sequence.
//
// "推测解码" (world.lapla.si/zh/specdec), section 通过的规则: with p the large
// model's and q the small model's probability of the guessed token, the
// guess is kept iff r <= p/q for a uniform r (so q <= p always keeps it).
// Section 留下对的，换掉错的: checking stops at the first guess that fails.
// Greedy mode (maxstudionews.com article 1664, the verify paragraph) keeps a
// guess iff it equals the large model's argmax.
//
// Each warp folds the per-tile partials of one row into (max, sum) -- the
// log-normaliser of z/T -- and the row's argmax; warp 0 then tests the
// gamma guesses in parallel and finds the first rejection with a ballot.
#include "accept.cuh"

namespace specdec {
namespace {

constexpr int kThreads = 512;   // one warp per record row: up to 2*32+1 rows in one round

template <typename DL>
__global__ void __launch_bounds__(kThreads) accept_kernel(const AcceptLaunch a) {
  __shared__ AcceptSmem sm;
  const int b = blockIdx.x;
  grid_dependency_wait();      // the LM-head kernel's records are complete
  grid_launch_dependents();    // the sampler may start launching
  if (b == 0 && threadIdx.x == 0) *a.calls += 1;   // the LM head of this call is done
  accept_fold<DL>(a, b, sm);
  __syncthreads();
  if (threadIdx.x >= 32) return;
  accept_decide<DL>(a, b, sm, true);
  if (threadIdx.x == 0 && a.mode == SPECDEC_SAMPLE) {
    a.sel[b] = sm.sr;
    a.counters[b] = 0;
  }
}

}  // namespace

cudaError_t launch_accept(const AcceptLaunch& L, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.B);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.dl_bf16) return cudaLaunchKernelEx(&cfg, accept_kernel<__nv_bfloat16>, L);
  return cudaLaunchKernelEx(&cfg, accept_kernel<float>, L);
}

}  // namespace specdec
