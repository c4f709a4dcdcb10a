"""The C-ABI library loads and exports every declared symbol; host-side logic and
argument validation (no GPU needed: nothing here reaches a CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import __graft_entry__ as entry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ft():
    entry.build()
    import expert_cache_gb300
    return expert_cache_gb300


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ft.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ft_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(ft):
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(ft.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ft.EXPORTED)


def test_record_bytes_match_oracle_layout(ft):
    from oracle.formats import record_layout
    for H, I in ((64, 32), (2048, 512), (4096, 2048), (128, 96)):
        assert ft.ft_record_bytes(H, I) == record_layout(H, I)["bytes"]
    with pytest.raises(ft.FtError):
        ft.ft_record_bytes(100, 32)


def test_split_helpers_match_oracle(ft):
    from oracle import qrule
    for _, bp, bh in [r for r in (l.split() for l in open(os.path.join(ROOT, "tests/golden/machine_bandwidths.txt")))
                      if r and not r[0].startswith("#")]:
        bp, bh = float(bp), float(bh)
        assert ft.ft_split_from_bandwidth(bp, bh) == qrule.split_from_bandwidth(bp, bh)
        assert ft.ft_split_from_overlap(bp, bh - bp) == qrule.split_from_overlap(bp, bh - bp)
    assert ft.ft_split_from_bandwidth(60, 50) == 65536
    assert ft.ft_split_from_bandwidth(0, 50) == 0 and ft.ft_split_from_overlap(-1, 2) == 0
    assert ft.ft_split_from_overlap(48, 40) == 35747


def _desc(ft, **kw):
    base = dict(L=2, E=16, H=64, I=32, k_max=2, B_max=1, capacity=8, capacity_max=0, T_max=0)
    base.update(kw)
    return ft.FtCacheDesc(base["L"], base["E"], base["H"], base["I"], base["k_max"], base["B_max"],
                          base["capacity"], base["capacity_max"], base["T_max"], None, None, None,
                          None, ft.FtSplit(ft.FT_SPLIT_FULL_OFFLOAD, 65536))


def test_required_sizes_and_validation(ft):
    rb, wb = ft.ft_cache_required_sizes(_desc(ft))
    assert rb == 3584 and wb > 0 and wb % 256 == 0
    _, wb2 = ft.ft_cache_required_sizes(_desc(ft, capacity_max=64))
    assert wb2 > wb
    for bad in (dict(E=0), dict(E=5000), dict(H=96), dict(I=48), dict(k_max=0), dict(B_max=33),
                dict(B_max=32, k_max=32), dict(capacity=0), dict(capacity=20000),
                dict(capacity=8, capacity_max=4), dict(L=0)):
        with pytest.raises(ft.FtError) as ei:
            ft.ft_cache_required_sizes(_desc(ft, **bad))
        assert ei.value.status == ft.FT_ERR_ARG
    d = _desc(ft)
    d.split = ft.FtSplit(ft.FT_SPLIT_QSTAR, 0)
    with pytest.raises(ft.FtError):
        ft.ft_cache_required_sizes(d)


def test_create_rejects_missing_memory(ft):
    with pytest.raises(ft.FtError) as ei:
        ft.ft_cache_create(_desc(ft))          # NULL pool / slots / workspace
    assert ei.value.status == ft.FT_ERR_ARG


def test_calls_on_null_handle(ft):
    with pytest.raises(ft.FtError):
        ft.ft_moe_decode(None, 0, 0, 0, 0, 1, 1, 0, 0, stream=0)
    with pytest.raises(ft.FtError):
        ft.ft_set_split(None, ft.FT_SPLIT_QSTAR, 100)
