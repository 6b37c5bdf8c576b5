"""Host logic of bench.py that decides what the JSON line may claim.

`roofline.traffic` comes from the committed ncu summary of the decode GEMV; it
must be dropped (None) whenever the kernel sources differ from the ones the
counters were taken on, and otherwise be the summary's own ratio."""
from __future__ import annotations

import re

import bench


def _profile_line():
    txt = open(bench.os.path.join(bench.ROOT, "profiles", "gemv_exl2_decode_70b.md")).read()
    m = re.search(r"bench-traffic: dram_bytes_per_algorithmic_byte=([0-9.]+) source_hash=([0-9a-f]+)", txt)
    assert m, "the decode profile carries a bench-traffic line"
    return float(m.group(1)), m.group(2)


def test_traffic_dropped_when_sources_differ(monkeypatch):
    monkeypatch.setattr(bench, "source_hash", lambda paths: "0" * 16)
    assert bench.profile_traffic() is None


def test_traffic_is_the_profiles_ratio_when_sources_match(monkeypatch):
    ratio, digest = _profile_line()
    monkeypatch.setattr(bench, "source_hash", lambda paths: digest)
    got = bench.profile_traffic()
    assert got == ratio
    # DRAM bytes can not be fewer than the packed bytes the kernel must read
    assert 1.0 <= got < 2.0


def test_source_hash_covers_the_gemv_sources():
    # every file the hash covers exists, and the hash changes with any of them
    assert bench.GEMV_SOURCES
    h = bench.source_hash(bench.GEMV_SOURCES)
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    assert bench.source_hash(bench.GEMV_SOURCES[:-1]) != h or len(bench.GEMV_SOURCES) == 1
