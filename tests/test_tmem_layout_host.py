"""CPU: the attention kernels' TMEM column maps, read from the sources.

Each kernel allocates all 512 TMEM columns and places its score (S), output
(O, d values plus the 16-column l block) and P regions at fixed columns; a
region that overlapped another would corrupt results only for some head
dims or in some tile orders.  These tests read the column constants from the
kernel sources and check that every region fits and that no two overlap, for
every head dim the kernels take (d = 8..128).
"""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc")
TMEM_COLS = 512


def _src(name):
    return open(os.path.join(CSRC, name)).read()


def _disjoint(regions):
    regions = sorted(regions)
    for (a, wa, na), (b, wb, nb) in zip(regions, regions[1:]):
        assert a + wa <= b, "%s [%d, %d) overlaps %s [%d, %d)" % (na, a, a + wa, nb, b, b + wb)
    for a, wa, n in regions:
        assert 0 <= a and a + wa <= TMEM_COLS, n


def _ocols(d):
    return ((d + 15) // 16) * 16 + 16     # d rounded to 16, plus the l block


def test_two_tile_maps():
    s = _src("attn_fp8_2tile.cu")
    m_s = re.search(r"tm_s\(int g\) \{ return OWN_S \? uint32_t\(g\) \* (\d+)u : (\d+)u; \}", s)
    m_o = re.search(r"tm_o\(int g\) \{ return OWN_S \? \(g \? (\d+)u : (\d+)u\) : \(g \? (\d+)u : (\d+)u\); \}", s)
    m_p = re.search(r"tm_p\(int g\) \{ return OWN_S \? \(g \? (\d+)u : (\d+)u\) : \(g \? (\d+)u : (\d+)u\); \}", s)
    own_max = int(re.search(r"constexpr int OWN_S_MAX_OCOLS = (\d+);", s).group(1))
    bn = int(re.search(r"constexpr int BN = (\d+);", s).group(1))
    assert m_s and m_o and m_p
    s_step, s_shared = int(m_s.group(1)), int(m_s.group(2))
    ob_own, oa_own, ob_sh, oa_sh = map(int, m_o.groups())
    pb_own, pa_own, pb_sh, pa_sh = map(int, m_p.groups())
    pcols = bn // 4                         # 4 E4M3 keys per 32-bit column
    for d in range(8, 129, 8):
        oc = _ocols(d)
        if oc <= own_max:                   # one S buffer per tile
            _disjoint([(0, bn, "S_A"), (s_step, bn, "S_B"), (oa_own, oc, "O_A"), (ob_own, oc, "O_B"),
                       (pa_own, pcols, "P_A"), (pb_own, pcols, "P_B")])
        # the shared-S layout is used above own_max but must hold every d
        _disjoint([(s_shared, bn, "S"), (oa_sh, oc, "O_A"), (ob_sh, oc, "O_B"),
                   (pa_sh, pcols, "P_A"), (pb_sh, pcols, "P_B")])
    assert _ocols(80) <= own_max < _ocols(96)   # d <= 80 gets one S buffer per tile


def test_one_tile_map():
    s = _src("attn_fp8.cu")
    m = re.search(r"constexpr uint32_t TM_S = (\d+), TM_O = (\d+), TM_P = (\d+);", s)
    bn = int(re.search(r"constexpr int BN = (\d+);", s).group(1))
    osplit = int(re.search(r"constexpr int OSPLIT = (\d+);", s).group(1))
    tm_s, tm_o, tm_p = map(int, m.groups())
    # O is read and rescaled as 2 x OSPLIT columns (two threads per row), so
    # that whole span must stay clear of P.
    assert 2 * osplit >= _ocols(128)
    _disjoint([(tm_s, bn, "S"), (tm_o, 2 * osplit, "O"), (tm_p, bn // 4, "P")])
