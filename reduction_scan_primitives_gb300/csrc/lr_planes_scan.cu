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

// Column-group runs (16 and 32 columns).
template <int P>
cudaError_t launch_cg_p(const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  const bool rev = (p.flags & kScanMirror) == 0;
  const bool excl = (p.flags & kScanExclusive) != 0;
  if (rev) {
    if (excl) launch_pdl(k_planes_cg<P, true, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_cg<P, true, false>, g, kT, 0, s, p);
  } else {
    if (excl) launch_pdl(k_planes_cg<P, false, true>, g, kT, 0, s, p);
    else launch_pdl(k_planes_cg<P, false, false>, g, kT, 0, s, p);
  }
  return cudaGetLastError();
}

template <int P>
int occupancy_cg_p() {
  return std::min({occupancy_of(k_planes_cg<P, false, false>), occupancy_of(k_planes_cg<P, false, true>),
                   occupancy_of(k_planes_cg<P, true, false>), occupancy_of(k_planes_cg<P, true, true>)});
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
    case 16: return launch_cg_p<16>(p, g, s);
    case 32: return launch_cg_p<32>(p, g, s);
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
    case 16: return occupancy_cg_p<16>();
    case 32: return occupancy_cg_p<32>();
    default: return 0;
  }
}

}  // namespace lr
