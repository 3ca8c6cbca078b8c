// lr_planes_lb.cu -- the look-back form for few long narrow planes
// (lr_planes.cuh): instantiations, launch and occupancy.
#include "lr_planes.cuh"

namespace lr {
namespace {

template <int P>
cudaError_t launch_lb_p(const PlaneLbParams& p, dim3 g, cudaStream_t s) {
  const bool rev = (p.flags & kScanMirror) == 0;
  const bool excl = (p.flags & kScanExclusive) != 0;
  if (rev) {
    if (excl) launch_pdl(k_planes_lb<P, true, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_lb<P, true, false>, g, kT, 0, s, p);
  } else {
    if (excl) launch_pdl(k_planes_lb<P, false, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_lb<P, false, false>, g, kT, 0, s, p);
  }
  return cudaGetLastError();
}

template <int P>
int occupancy_lb_p() {
  return std::min({occupancy_of(k_planes_lb<P, false, false>), occupancy_of(k_planes_lb<P, false, true>),
                   occupancy_of(k_planes_lb<P, true, false>), occupancy_of(k_planes_lb<P, true, true>)});
}

// Column groups (6 .. 128 columns), instances as the column-group scans.
template <int V, int GMAX, int GFIX>
cudaError_t launch_cg_lb_v(const PlaneLbParams& p, dim3 g, cudaStream_t s) {
  const bool rev = (p.flags & kScanMirror) == 0;
  const bool excl = (p.flags & kScanExclusive) != 0;
  if (rev) {
    if (excl) launch_pdl(k_planes_cg_lb<V, GMAX, GFIX, true, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_cg_lb<V, GMAX, GFIX, true, false>, g, kT, 0, s, p);
  } else {
    if (excl) launch_pdl(k_planes_cg_lb<V, GMAX, GFIX, false, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_cg_lb<V, GMAX, GFIX, false, false>, g, kT, 0, s, p);
  }
  return cudaGetLastError();
}

template <int V, int GMAX, int GFIX>
int occupancy_cg_lb_v() {
  return std::min({occupancy_of(k_planes_cg_lb<V, GMAX, GFIX, false, false>),
                   occupancy_of(k_planes_cg_lb<V, GMAX, GFIX, false, true>),
                   occupancy_of(k_planes_cg_lb<V, GMAX, GFIX, true, false>),
                   occupancy_of(k_planes_cg_lb<V, GMAX, GFIX, true, true>)});
}

}  // namespace

cudaError_t launch_planes_cg_lookback(const PlaneLbParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (cg_instance(p.P)) {
    case 0: return launch_cg_lb_v<1, 32, 0>(p, g, s);
    case 1: return launch_cg_lb_v<2, 32, 0>(p, g, s);
    case 2: return launch_cg_lb_v<4, 8, 0>(p, g, s);
    case 3: return launch_cg_lb_v<4, 32, 0>(p, g, s);
    case 4: return launch_cg_lb_v<4, 8, 4>(p, g, s);
    case 5: return launch_cg_lb_v<4, 8, 8>(p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes_cg_lookback(int instance) {
  switch (instance) {
    case 0: return occupancy_cg_lb_v<1, 32, 0>();
    case 1: return occupancy_cg_lb_v<2, 32, 0>();
    case 2: return occupancy_cg_lb_v<4, 8, 0>();
    case 3: return occupancy_cg_lb_v<4, 32, 0>();
    case 4: return occupancy_cg_lb_v<4, 8, 4>();
    case 5: return occupancy_cg_lb_v<4, 8, 8>();
    default: return 0;
  }
}

cudaError_t launch_planes_lookback(int P, const PlaneLbParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (P) {
    case 2: return launch_lb_p<2>(p, g, s);
    case 3: return launch_lb_p<3>(p, g, s);
    case 4: return launch_lb_p<4>(p, g, s);
    case 5: return launch_lb_p<5>(p, g, s);
    case 6: return launch_lb_p<6>(p, g, s);
    case 7: return launch_lb_p<7>(p, g, s);
    case 8: return launch_lb_p<8>(p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes_lookback(int P) {
  switch (P) {
    case 2: return occupancy_lb_p<2>();
    case 3: return occupancy_lb_p<3>();
    case 4: return occupancy_lb_p<4>();
    case 5: return occupancy_lb_p<5>();
    case 6: return occupancy_lb_p<6>();
    case 7: return occupancy_lb_p<7>();
    case 8: return occupancy_lb_p<8>();
    default: return 0;
  }
}

}  // namespace lr
