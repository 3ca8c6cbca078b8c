// lr_planes_reduce.cu -- the reductions of narrow planes (lr_planes.cuh):
// instantiations, launch and occupancy.
#include "lr_planes.cuh"

namespace lr {
namespace {

template <int P, bool MULTI>
cudaError_t launch_reduce_pm(int op, const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  switch (op) {
    case kOpSum: launch_pdl(k_planes<P, false, false, false, OpSum, MULTI>, g, kT, 0, s, p); break;
    case kOpSumSq: launch_pdl(k_planes<P, false, false, false, OpSumSq, MULTI>, g, kT, 0, s, p); break;
    case kOpMax: launch_pdl(k_planes<P, false, false, false, OpMax, MULTI>, g, kT, 0, s, p); break;
    case kOpMin: launch_pdl(k_planes<P, false, false, false, OpMin, MULTI>, g, kT, 0, s, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int P>
cudaError_t launch_reduce_p(int op, const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  return p.multi ? launch_reduce_pm<P, true>(op, p, g, s) : launch_reduce_pm<P, false>(op, p, g, s);
}

template <int P>
int occupancy_reduce_p() {
  return std::min(occupancy_of(k_planes<P, false, false, false, OpSum, false>),
                  occupancy_of(k_planes<P, false, false, false, OpSum, true>));
}

// Column groups (9 .. 128 columns).
template <int V, int GMAX, int GFIX>
cudaError_t launch_cg_reduce_v(int op, const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  switch (op) {
    case kOpSum: launch_pdl(k_planes_cg_reduce<V, GMAX, GFIX, OpSum>, g, kT, 0, s, p); break;
    case kOpSumSq: launch_pdl(k_planes_cg_reduce<V, GMAX, GFIX, OpSumSq>, g, kT, 0, s, p); break;
    case kOpMax: launch_pdl(k_planes_cg_reduce<V, GMAX, GFIX, OpMax>, g, kT, 0, s, p); break;
    case kOpMin: launch_pdl(k_planes_cg_reduce<V, GMAX, GFIX, OpMin>, g, kT, 0, s, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int V, int GMAX, int GFIX>
int occupancy_cg_reduce_v() {
  return std::min({occupancy_of(k_planes_cg_reduce<V, GMAX, GFIX, OpSum>),
                   occupancy_of(k_planes_cg_reduce<V, GMAX, GFIX, OpSumSq>),
                   occupancy_of(k_planes_cg_reduce<V, GMAX, GFIX, OpMax>),
                   occupancy_of(k_planes_cg_reduce<V, GMAX, GFIX, OpMin>)});
}

}  // namespace

cudaError_t launch_planes_cg_reduce(int op, const PlaneRunParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (cg_instance(p.P)) {
    case 0: return launch_cg_reduce_v<1, 32, 0>(op, p, g, s);
    case 1: return launch_cg_reduce_v<2, 32, 0>(op, p, g, s);
    case 2: return launch_cg_reduce_v<4, 8, 0>(op, p, g, s);
    case 3: return launch_cg_reduce_v<4, 32, 0>(op, p, g, s);
    case 4: return launch_cg_reduce_v<4, 8, 4>(op, p, g, s);
    case 5: return launch_cg_reduce_v<4, 8, 8>(op, p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes_cg_reduce(int instance) {
  switch (instance) {
    case 0: return occupancy_cg_reduce_v<1, 32, 0>();
    case 1: return occupancy_cg_reduce_v<2, 32, 0>();
    case 2: return occupancy_cg_reduce_v<4, 8, 0>();
    case 3: return occupancy_cg_reduce_v<4, 32, 0>();
    case 4: return occupancy_cg_reduce_v<4, 8, 4>();
    case 5: return occupancy_cg_reduce_v<4, 8, 8>();
    default: return 0;
  }
}

cudaError_t launch_planes_reduce(int P, int op, const PlaneRunParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (P) {
    case 2: return launch_reduce_p<2>(op, p, g, s);
    case 3: return launch_reduce_p<3>(op, p, g, s);
    case 4: return launch_reduce_p<4>(op, p, g, s);
    case 5: return launch_reduce_p<5>(op, p, g, s);
    case 6: return launch_reduce_p<6>(op, p, g, s);
    case 7: return launch_reduce_p<7>(op, p, g, s);
    case 8: return launch_reduce_p<8>(op, p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes_reduce(int P) {
  switch (P) {
    case 2: return occupancy_reduce_p<2>();
    case 3: return occupancy_reduce_p<3>();
    case 4: return occupancy_reduce_p<4>();
    case 5: return occupancy_reduce_p<5>();
    case 6: return occupancy_reduce_p<6>();
    case 7: return occupancy_reduce_p<7>();
    case 8: return occupancy_reduce_p<8>();
    default: return 0;
  }
}

}  // namespace lr
