"""Host-side arithmetic of bench.py (CPU only): the algorithmic byte and FMA
counts behind its roofline fractions, and the digest gate on recorded DRAM
traffic."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_of_the_headline_call(bench):
    # int4 [12288, 6144], S = 1: codes 12288 * 3072 + scales 4 * 12288 + x 4 * 6144 + y 4 * 12288
    assert bench.algorithmic_bytes(4, 12288, 6144, 1) == 12288 * 3072 + 4 * 12288 + 4 * 6144 + 4 * 12288
    assert bench.algorithmic_bytes(4, 12288, 6144, 1) == 37871616
    # ragged rows: ceil(I * bits / 8) bytes per row
    assert bench.algorithmic_bytes(2, 3, 5, 2) == 3 * 2 + 4 * 3 + 4 * 2 * 5 + 4 * 2 * 3
    assert bench.algorithmic_bytes(32, 2, 3, 1) == 2 * 12 + 8 + 12 + 8


def _mla_fma_by_steps(H, Dn, Dv, K, R, S, T, st0):
    """Multiply-adds of the four steps, counted one (head, token) at a time."""
    n = 0
    for _h in range(H):
        for s in range(S):
            window = (T - S + s) - st0 + 1
            n += Dn * K             # absorb: qabs from Dn key rows of K columns
            n += window * (K + R)   # scores over latent and rope
            n += window * K         # latent context
            n += Dv * K             # value rows
    return n


@pytest.mark.parametrize("H,Dn,Dv,K,R,S,T,st0", [(64, 128, 128, 512, 64, 1, 4096, 0), (3, 8, 5, 40, 8, 4, 70, 7),
                                                 (2, 4, 4, 16, 0, 1, 1, 0), (5, 7, 9, 132, 12, 2, 33, 31)])
def test_mla_fma_count(bench, H, Dn, Dv, K, R, S, T, st0):
    assert bench.mla_fma(H, Dn, Dv, K, R, S, T, st0) == _mla_fma_by_steps(H, Dn, Dv, K, R, S, T, st0)


def test_mla_bytes(bench):
    # caches of the window, int4 codes + f32 row scales, q_nope + q_rope + ctx
    H, Dn, Dv, K, R, S, T = 64, 128, 128, 512, 64, 1, 4096
    rows = H * (Dn + Dv)
    assert bench.mla_bytes(H, Dn, Dv, K, R, S, T) == T * (K + R) * 4 + rows * (K // 2 + 4) + S * H * (Dn + R + Dv) * 4


def test_recorded_traffic_needs_the_current_source(bench, tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// one kernel\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.source_digest(["kernel.cu"])
    table = tmp_path / "traffic.txt"
    table.write_text("# comment line\nkey=k1 sources=kernel.cu digest=%s bytes_per_launch=1234\n" % digest)
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(table))
    assert bench.recorded_traffic("k1") == 1234.0
    assert bench.recorded_traffic("other") is None
    src.write_text("// one kernel, changed\n")                  # the capture no longer describes the source
    assert bench.recorded_traffic("k1") is None


def test_committed_traffic_records_name_existing_sources(bench):
    for ln in open(bench.TRAFFIC_FILE).read().splitlines():
        if ln.startswith("key="):
            kv = dict(p.split("=", 1) for p in ln.split())
            for f in kv["sources"].split(","):
                assert os.path.exists(os.path.join(ROOT, f)), f
            assert float(kv["bytes_per_launch"]) > 0


def test_cpu_model_and_oracle_timer(bench):
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
    calls = []
    n, dt = bench.time_oracle(lambda: calls.append(1), 0.01, min_calls=3)
    assert n >= 3 and dt >= 0.01 and len(calls) == n + 1    # one untimed warm call
