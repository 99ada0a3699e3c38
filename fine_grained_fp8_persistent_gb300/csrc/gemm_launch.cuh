// gemm_launch.cuh -- host side of one GEMM launch: tensor maps, the tile-shape
// heuristic, persistent grid sizing and the cluster launch.
#pragma once
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "gemm_persistent.cuh"

namespace fgf8 {

// One kernel configuration the launchers can choose from.
struct TileCfg {
  int ncta;       // 1 = one CTA per tile, 2 = a CTA pair per tile (M = 256)
  int bn;         // tile width
  double t_tile;  // relative time of one cluster tile (measured, see pick_cfg)
  bool ws = false;  // weight-stationary: one CTA, 256 rows as two .ws sub-tiles
};

// Entries of a candidate table.
template <int N>
constexpr int kCount(const TileCfg (&)[N]) { return N; }

// Tiles of the problem for a configuration, counted per cluster (masked and
// contiguous pairs: upper bounds).
inline long long tile_count(const GemmArgs& a, Sched s, const TileCfg& c) {
  const long long tm = 128LL * c.ncta * (c.ws ? 2 : 1);
  long long mt = (a.M + tm - 1) / tm;
  if (s == Sched::Contiguous && c.ncta == 2) {
    // pairs are cut per expert segment: each segment may end on half a pair
    const long long blocks = (a.M + 127) / 128;
    mt = (blocks + (a.G < blocks ? a.G : blocks) + 1) / 2;
  }
  const long long nt = (a.N + c.bn - 1) / c.bn;
  return (s == Sched::Masked ? a.G : 1) * mt * nt;
}

// Estimated time of a configuration: waves of cluster tiles over the SMs times the
// time of one cluster tile.  The tile times are measured on a GB300 at M = 4096,
// N = K = 7168 (microseconds per tile, the same K for every candidate, so only
// their ratios matter); the widths not measured there are extrapolated from the
// narrowest measured ones.  A wide tile wins on large problems; narrow tiles spread
// skinny problems over more SMs (the DeepGEMM page's unaligned BLOCK_N argument:
// 112 vs 128 blocks on 132 SMs).
// FGF8_FORCE_TILE="<ctas per cluster>x<bn>[ws]" (e.g. "2x224", "1x128", "1x128ws")
// selects that configuration when it is among the candidates (used by the tests to
// cover every instantiation).
inline int pick_cfg(const GemmArgs& a, Sched s, const TileCfg* cands, int n) {
  if (const char* f = std::getenv("FGF8_FORCE_TILE")) {
    int nc = 0, bn = 0;
    char suffix[4] = {0, 0, 0, 0};
    const int got = std::sscanf(f, "%dx%d%3s", &nc, &bn, suffix);
    const bool ws = got == 3 && std::strcmp(suffix, "ws") == 0;
    if (got >= 2)
      for (int i = 0; i < n; ++i)
        if (cands[i].ncta == nc && cands[i].bn == bn && cands[i].ws == ws) return i;
  }
  const long long sms = device_sm_count();
  int best = 0;
  double best_cost = -1.0;
  for (int i = 0; i < n; ++i) {
    const long long units = sms / cands[i].ncta;
    const long long waves = (tile_count(a, s, cands[i]) + units - 1) / units;
    const double cost = static_cast<double>(waves) * cands[i].t_tile;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = i;
    }
  }
  return best;
}

// Contiguous layout on CTA pairs: the scheduler keeps one entry per expert
// segment in shared memory, for at most this many 128-row blocks.
constexpr int kMaxContiguousPairBlocks = 512;

// Largest dynamic shared memory a CTA may opt into on sm_100-class parts (227 KB).
constexpr int kMaxSmemOptin = 232448;

template <Kind KIND, Sched SCHED, int NCTA, int BN, int STAGES, int NACC = 2, int AROWS = 128,
          bool QOUT = false>
int launch_persistent(const GemmArgs& a, const TensorMaps& tm, long long tiles, cudaStream_t stream) {
  using C = PCfg<KIND, SCHED, NCTA, BN, STAGES, NACC, AROWS, QOUT>;
  static_assert(C::SMEM_BYTES <= kMaxSmemOptin, "shared memory budget");
  auto* fn = &gemm_persistent<KIND, SCHED, NCTA, BN, STAGES, NACC, AROWS, QOUT>;
  if ((a.dq != nullptr) != QOUT) return set_error(2, "output quantization and kernel disagree");
  constexpr int CL = C::CLUSTER;
  static int max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return set_error(2, "device id %d", dev);
  if (C::SMEM_BYTES > device_max_smem_optin())
    return set_error(2, "tile needs %d bytes of shared memory", C::SMEM_BYTES);
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return set_error(4, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    int clusters = 0;
    cfg.gridDim = dim3(CL * (device_sm_count() / CL), 1, 1);
    // the CTAs of a cluster are co-scheduled inside one GPC, so the number of pairs
    // that fit can be below SMs / 2 ("Dissecting NVIDIA Blackwell" (EEPW), section
    // on clusters, GPCs and die yield)
    e = CL > 1 ? cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) : cudaSuccess;
    if (CL == 1) clusters = device_sm_count();
    if (e != cudaSuccess || clusters <= 0)
      return set_error(4, "cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
    max_clusters[dev] = clusters;
  }
  // static schedule: a persistent grid, capped for dense GEMMs by the wave-preserving
  // SM count (grouped layouts only know an upper bound of their tiles here); cluster
  // launch control: one cluster per tile, the kernel cancels the clusters that have
  // not launched yet and takes their tiles
  GemmArgs la = a;
  la.clc = scheduler_mode();
  long long clc_tiles = tiles;
  if (SCHED == Sched::Contiguous && CL == 2) {
    // pairs are cut per run of same-expert blocks on the device: at most one pair
    // tile per 128-row block, whatever the runs (a bound that holds for any m_indices)
    clc_tiles = static_cast<long long>((a.M + 127) / 128) * ((a.N + BN - 1) / BN);
  }
  long long clusters = la.clc ? (clc_tiles > 0 ? clc_tiles : 1)
                              : persistent_clusters(tiles, CL, device_sm_count(), max_clusters[dev],
                                                    SCHED == Sched::Dense && sm_cap_enabled());
  if (clusters * CL > 0x7FFFFFFFLL) return set_error(2, "gemm launch: %lld tiles exceed the grid limit", tiles);
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL), 1, 1);
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  set_last_tile(KIND == Kind::F16    ? "f16"
                : KIND == Kind::MXF8 ? "mxf8"
                : KIND == Kind::MXF4 ? "mxf4"
                : KIND == Kind::NVF4 ? "nvf4"
                                     : "f8f32",
                SCHED == Sched::Dense ? "dense" : SCHED == Sched::Contiguous ? "contiguous" : "masked", CL, BN,
                C::kWS ? "ws" : "");
  // the output map of the TMA-store epilogue: 32 x 32 boxes of 16-bit values
  CUtensorMap tm_d;
  std::memset(&tm_d, 0, sizeof(tm_d));
  if constexpr (C::kTmaStore) {
    // rows of D: M (dense, contiguous) or G x Mmax (masked, experts stacked)
    const uint64_t d_rows = static_cast<uint64_t>(a.M) * (SCHED == Sched::Masked ? static_cast<uint64_t>(a.G) : 1u);
    if (!encode_tmap_2d(&tm_d, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.D, static_cast<uint64_t>(a.N), d_rows,
                        static_cast<uint64_t>(a.N) * 2u, 32, 32, false))
      return 4;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, tm.a, tm.b, tm.sfa, tm.sfb, tm_d, la);
  if (e != cudaSuccess) return set_error(4, "gemm launch: %s", cudaGetErrorString(e));
  return 0;
}

// Rows of a thin tile's A box: M rounded up to 8, at most the 64-row stage.  A
// box reaching far past the M rows of A costs time in the copy engine (with
// 64-row boxes the M = 1 decode at N = K = 7168 took 28.3 us against 18.8 us at
// M = 64); the stage rows past the box feed only accumulator rows that are never
// stored.
inline int thin_a_box_rows(int M) { return M >= 64 ? 64 : (M + 7) / 8 * 8; }

// A and B operand maps: K-major rows of 128 bytes per stage, 128-byte swizzle;
// each CTA loads 128 rows of A and BN / NCTA rows of B.
inline int make_operand_maps(TensorMaps& tm, CUtensorMapDataType dt, int elem_bytes, const void* A,
                             long long a_rows, const void* B, long long b_rows, int K, int b_box_rows,
                             int a_box_rows = 128) {
  std::memset(&tm, 0, sizeof(tm));
  const uint32_t bk = 128 / elem_bytes;
  if (!encode_tmap_2d(&tm.a, dt, A, K, a_rows, static_cast<uint64_t>(K) * elem_bytes, bk, a_box_rows, true))
    return 4;
  if (!encode_tmap_2d(&tm.b, dt, B, K, b_rows, static_cast<uint64_t>(K) * elem_bytes, bk, b_box_rows,
                      true))
    return 4;
  return 0;
}

}  // namespace fgf8
