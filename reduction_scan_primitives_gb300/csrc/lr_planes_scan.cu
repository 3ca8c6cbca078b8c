// lr_planes_scan.cu -- the scans of narrow planes (lr_planes.cuh): instantiations,
// launch and occupancy.
#include "lr_planes.cuh"

namespace lr {
namespace {

template <int P, bool REV, bool MULTI>
cudaError_t launch_scan_dir(const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  if (p.flags & kScanExclusive) launch_pdl(k_planes<P, true, REV, true, OpSum, MULTI>, g, kT, 0, s, p);
  else launch_pdl(k_planes<P, true, REV, false, OpSum, MULTI>, g, kT, 0, s, p);
  return cudaGetLastError();
}

template <int P>
cudaError_t launch_scan_p(const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  if (p.multi)
    return (p.flags & kScanMirror) ? launch_scan_dir<P, false, true>(p, g, s) : launch_scan_dir<P, true, true>(p, g, s);
  return (p.flags & kScanMirror) ? launch_scan_dir<P, false, false>(p, g, s) : launch_scan_dir<P, true, false>(p, g, s);
}

template <int P>
int occupancy_scan_p() {
  return std::min({occupancy_of(k_planes<P, true, false, false, OpSum, false>),
                   occupancy_of(k_planes<P, true, false, true, OpSum, false>),
                   occupancy_of(k_planes<P, true, true, false, OpSum, false>),
                   occupancy_of(k_planes<P, true, true, true, OpSum, false>),
                   occupancy_of(k_planes<P, true, false, false, OpSum, true>),
                   occupancy_of(k_planes<P, true, true, true, OpSum, true>)});
}

// Column groups (any other column count up to 128).
template <int V, int GMAX, int GFIX>
cudaError_t launch_cg_v(const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  const bool rev = (p.flags & kScanMirror) == 0;
  const bool excl = (p.flags & kScanExclusive) != 0;
  if (rev) {
    if (excl) launch_pdl(k_planes_cg<V, GMAX, GFIX, true, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_cg<V, GMAX, GFIX, true, false>, g, kT, 0, s, p);
  } else {
    if (excl) launch_pdl(k_planes_cg<V, GMAX, GFIX, false, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_cg<V, GMAX, GFIX, false, false>, g, kT, 0, s, p);
  }
  return cudaGetLastError();
}

template <int V, int GMAX, int GFIX>
int occupancy_cg_v() {
  return std::min({occupancy_of(k_planes_cg<V, GMAX, GFIX, false, false>),
                   occupancy_of(k_planes_cg<V, GMAX, GFIX, false, true>),
                   occupancy_of(k_planes_cg<V, GMAX, GFIX, true, false>),
                   occupancy_of(k_planes_cg<V, GMAX, GFIX, true, true>)});
}

}  // namespace

cudaError_t launch_planes_scan(int P, const PlaneRunParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (P) {
    case 2: return launch_scan_p<2>(p, g, s);
    case 3: return launch_scan_p<3>(p, g, s);
    case 4: return launch_scan_p<4>(p, g, s);
    case 5: return launch_scan_p<5>(p, g, s);
    case 6: return launch_scan_p<6>(p, g, s);
    case 7: return launch_scan_p<7>(p, g, s);
    case 8: return launch_scan_p<8>(p, g, s);
    case 9: return launch_scan_p<9>(p, g, s);
    case 10: return launch_scan_p<10>(p, g, s);
    case 12: return launch_scan_p<12>(p, g, s);
    case 14: return launch_scan_p<14>(p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes(int P, bool scan) {
  if (!scan) return occupancy_planes_reduce(P);
  switch (P) {
    case 2: return occupancy_scan_p<2>();
    case 3: return occupancy_scan_p<3>();
    case 4: return occupancy_scan_p<4>();
    case 5: return occupancy_scan_p<5>();
    case 6: return occupancy_scan_p<6>();
    case 7: return occupancy_scan_p<7>();
    case 8: return occupancy_scan_p<8>();
    case 9: return occupancy_scan_p<9>();
    case 10: return occupancy_scan_p<10>();
    case 12: return occupancy_scan_p<12>();
    case 14: return occupancy_scan_p<14>();
    default: return 0;
  }
}

// The column-group instance for P columns: 0 .. 3 for (V, GMAX) = (1, 32),
// (2, 32), (4, 8), (4, 32) with the group count taken at run time, 4 and 5
// for 16 and 32 columns (4 and 8 float4 groups fixed at compile time); -1
// when P does not fit.
int cg_instance(int P) {
  if (!planes_cg_fits(P)) return -1;
  if (P == 16 || P == 32) return P == 16 ? 4 : 5;
  const int V = planes_cg_vec(P);
  return V == 1 ? 0 : V == 2 ? 1 : planes_cg_groups(P) <= 8 ? 2 : 3;
}

cudaError_t launch_planes_cg(const PlaneRunParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (cg_instance(p.P)) {
    case 0: return launch_cg_v<1, 32, 0>(p, g, s);
    case 1: return launch_cg_v<2, 32, 0>(p, g, s);
    case 2: return launch_cg_v<4, 8, 0>(p, g, s);
    case 3: return launch_cg_v<4, 32, 0>(p, g, s);
    case 4: return launch_cg_v<4, 8, 4>(p, g, s);
    case 5: return launch_cg_v<4, 8, 8>(p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes_cg(int instance) {
  switch (instance) {
    case 0: return occupancy_cg_v<1, 32, 0>();
    case 1: return occupancy_cg_v<2, 32, 0>();
    case 2: return occupancy_cg_v<4, 8, 0>();
    case 3: return occupancy_cg_v<4, 32, 0>();
    case 4: return occupancy_cg_v<4, 8, 4>();
    case 5: return occupancy_cg_v<4, 8, 8>();
    default: return 0;
  }
}

}  // namespace lr
