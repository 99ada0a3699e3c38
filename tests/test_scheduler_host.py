"""CPU checks of the launcher's grid rule for the static persistent schedule: the
wave-preserving SM cap ("DeepGEMM dissected", section on the number of SMs
launched: num_min_sms = ceil(max(SMs the waves need, SMs - 8) / multicast) *
multicast), checked against a brute-force search written from its definition."""
import ctypes
import math

import pytest


@pytest.fixture(scope="module")
def lib():
    from fine_grained_fp8_persistent_gb300 import build
    lib = ctypes.CDLL(build.build())
    lib.fgf8_persistent_clusters.argtypes = [ctypes.c_longlong, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int]
    lib.fgf8_persistent_clusters.restype = ctypes.c_longlong
    return lib


def brute_force(tiles, cluster, sms, max_clusters):
    """The fewest clusters that finish `tiles` in the same number of waves as the
    full grid, raised to at least (sms - 8) SMs' worth of whole clusters and kept
    within the full grid."""
    full = min(tiles, max_clusters)
    waves = math.ceil(tiles / full)
    fewest = min(c for c in range(1, full + 1) if math.ceil(tiles / c) == waves)
    floor_clusters = math.ceil((sms - 8) / cluster)
    return min(max(fewest, floor_clusters), full)


CASES = [
    (512, 2, 152, 76),      # 4096 x 7168 on 256 x 224 pair tiles: 6.74 waves -> 7 on 74 pairs
    (150, 1, 152, 152),     # the M = 64 decode on 48-wide tiles: one wave
    (1000, 1, 152, 152),    # 7 waves; the (SMs - 8) floor decides
    (304, 2, 152, 76),      # 16-bit 4096^3 on 256 x 224 tiles: exactly 4 waves
    (1, 2, 152, 74),
    (76, 2, 152, 74),       # fewer pairs fit than SMs / 2 (GPC packing)
    (3584, 1, 152, 152),
    (7, 1, 152, 152),
]


@pytest.mark.parametrize("tiles,cluster,sms,max_clusters", CASES)
def test_cap_matches_the_rule(lib, tiles, cluster, sms, max_clusters):
    got = lib.fgf8_persistent_clusters(tiles, cluster, sms, max_clusters, 1)
    assert got == brute_force(tiles, cluster, sms, max_clusters)
    # the cap never changes the number of waves
    full = min(tiles, max_clusters)
    assert math.ceil(tiles / got) == math.ceil(tiles / full)


@pytest.mark.parametrize("tiles,cluster,sms,max_clusters", CASES)
def test_without_cap_the_grid_is_full(lib, tiles, cluster, sms, max_clusters):
    assert lib.fgf8_persistent_clusters(tiles, cluster, sms, max_clusters, 0) == min(tiles, max_clusters)


def test_headline_values(lib):
    # the pages' formula by hand for the 512-tile case: waves = 7, SMs the waves
    # need = ceil(512 / 7) * 2 = 148, max(148, 152 - 8) = 148 -> 74 pairs
    assert lib.fgf8_persistent_clusters(512, 2, 152, 76, 1) == 74
    assert lib.fgf8_persistent_clusters(1000, 1, 152, 152, 1) == 144
