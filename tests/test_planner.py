"""Host-side checks of the skinny kernel's planner (no GPU needed).

tests/planner_check.cu compiles the planner (bit_weight_quantized_gb300/csrc/
gemv.cu) into a host program that prints each plan.  The plans must cover
every row and every K chunk, keep the padded pitch that makes the MMA quads'
reads conflict-free, lay out shared memory without overlap inside the per-CTA
limit, and fit the decode shapes in half an SM (two CTAs per SM, so that
consecutive calls overlap).

tests/decode_route_check.cu does the same for the decode kernel's shape rule
(bit_weight_quantized_gb300/csrc/decode.cu, decode_supports), checked against
the rule as documented for qmm_gemv.
"""
import json
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
KMAX_RING = 16


def _ceil(a, b):
    return (a + b - 1) // b


def _shapes():
    s = []
    s += [(1, 4096, 4096, b, 128, 0) for b in range(1, 9)]                 # decode sweep
    s += [(1, 512, 512, 4, 128, 0)]                                         # parity reference
    s += [(m, n, 4096, b, 64, 1) for m in (2, 4, 8, 16) for n in (11008, 14336)
          for b in (3, 4, 5, 6)]                                            # skinny batched decode
    s += [(m, 4096, 4096, 4, 128, 0) for m in (1, 16, 32, 64)]              # W4A8 shapes
    for b in range(1, 9):                                                   # edges
        for g in (32, 64, 128):
            s += [(1, 1, g, b, g, 1), (3, 130, 96 if g == 32 else 2 * g, b, g, 0),
                  (16, 15, 16384, b, g, 1), (9, 20000, 1024, b, g, 0), (16, 19800, 8192, b, g, 0),
                  (5, 152 * 128 + 7, 512, b, g, 1)]
    s += [(64, 20000, 1024, 4, 128, 0), (64, 4096, 65536, 4, 128, 0), (16, 4096, 65536, 8, 32, 1)]
    return s


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("planner") / "planner_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    "--expt-relaxed-constexpr", "-o", exe, os.path.join(HERE, "planner_check.cu")],
                   check=True, capture_output=True)
    shapes = _shapes()
    stdin = "".join(f"{m} {n} {k} {b} {g} {z}\n" for m, n, k, b, g, z in shapes)
    out = subprocess.run([exe], input=stdin, capture_output=True, text=True, check=True).stdout
    res = [json.loads(line) for line in out.splitlines()]
    assert len(res) == len(shapes)
    return res


def test_plans_exist(plans):
    bad = [(p["M"], p["N"], p["K"], p["bits"], p["group"]) for p in plans if p["st"] != 0]
    assert not bad, f"no plan for {bad}"


def test_rows_and_chunks_covered(plans):
    for p in plans:
        g, n = p["grid"], p["N"]
        assert 1 <= g <= p["num_sms"]
        assert p["rows_base"] * g + p["rows_rem"] == n and 0 <= p["rows_rem"] < g
        rows_max = p["rows_base"] + (1 if p["rows_rem"] else 0)
        assert 1 <= p["rb"] <= min(128, rows_max) and p["rbp"] == _ceil(p["rb"], 16) * 16
        assert p["nchunks"] == _ceil(p["K"], 128)
        assert p["stages_per_block"] == _ceil(p["nchunks"], p["seg_chunks"])
        assert p["nphases"] == _ceil(p["nchunks"], p["phase_chunks"])
        # a stage never straddles two activation phases
        assert p["nphases"] == 1 or p["phase_chunks"] % p["seg_chunks"] == 0


def test_segment_pitch_and_stage(plans):
    for p in plans:
        b = p["bits"]
        assert p["seg_bytes"] == p["seg_chunks"] * 16 * b
        assert p["pitch"] >= p["seg_bytes"] and p["pitch"] % 16 == 0
        # quad-strided reads of a tile's eight rows hit distinct banks
        assert p["pitch"] % 128 == (16 if b == 8 else 16 * b % 128)
        assert p["stage_bytes"] >= p["rb"] * p["pitch"] and p["stage_bytes"] % 128 == 0
        assert 1 <= p["ring"] <= KMAX_RING


def test_shared_memory_layout(plans):
    for p in plans:
        m, mp = p["M"], 8 * (1 if p["M"] <= 8 else 2 if p["M"] <= 16 else 4 if p["M"] <= 32 else 8)
        ngc = 128 // p["group"]
        ksplit = 1 << p["ksplit_log2"]
        x_need = m * p["phase_chunks"] * 128 * 2
        xs_need = p["phase_chunks"] * ngc * mp * 4
        sz_need = p["rbp"] * p["sz_pitch"] * ((2 + p["zeros"]) if p["sz_compact"] else 8)
        red_need = ksplit * p["rbp"] * mp * 4
        assert p["off_bar"] == 0 and p["off_x"] >= KMAX_RING * 12
        assert p["off_xs"] - p["off_x"] >= x_need
        assert p["off_cs"] - p["off_xs"] >= xs_need and p["off_sz"] - p["off_cs"] >= xs_need
        assert p["sz_pitch"] % 2 == 1 and p["sz_pitch"] >= p["K"] // p["group"]
        assert p["sz_compact"] == (1 if m > 8 else 0)
        if p["red_alias"]:
            assert p["off_red"] == p["off_x"] and red_need <= p["off_xs"] - p["off_x"]
            assert p["off_ring"] - p["off_sz"] >= sz_need
        else:
            assert p["off_red"] - p["off_sz"] >= sz_need
            assert p["off_ring"] - p["off_red"] >= red_need
        assert p["off_ring"] % 128 == 0
        # the ring, 128 bytes of read overrun, and the base-alignment slack
        assert p["off_ring"] + p["ring"] * p["stage_bytes"] + 128 + 128 <= p["smem"] <= p["smem_max"]


def test_decode_shapes_fit_two_ctas_per_sm(plans):
    for p in plans:
        if p["M"] == 1 and p["N"] == 4096 and p["K"] == 4096:
            assert p["smem"] <= p["smem_pair"], (p["bits"], p["smem"])


# ---- the decode kernel's shape rule (decode.cu) ------------------------------------
def _decode_rule(M, N, K, G, sms):
    """M <= 8, G in {64, 128}, K a positive multiple of 8 G, at most 32 columns per CTA
    with min(N, SMs) CTAs."""
    grid = min(N, sms)
    return 1 <= M <= 8 and G in (64, 128) and K >= 8 * G and K % (8 * G) == 0 and -(-N // grid) <= 32


def test_decode_route_rule(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "decode_route_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    "--expt-relaxed-constexpr", "-o", exe, os.path.join(HERE, "decode_route_check.cu")],
                   check=True, capture_output=True)
    shapes = [(M, N, K, G, sms) for M in (0, 1, 8, 9, 16) for G in (32, 64, 128)
              for K in (256, 512, 1024, 1536, 4096, 12288)
              for N in (1, 151, 152, 4096, 4863, 4864, 4865, 14336)
              for sms in (152, 148)]
    stdin = "".join(" ".join(map(str, s)) + "\n" for s in shapes)
    out = subprocess.run([exe], input=stdin, capture_output=True, text=True, check=True).stdout
    rows = [tuple(map(int, line.split())) for line in out.splitlines()]
    assert len(rows) == len(shapes)
    for r in rows:
        assert bool(r[5]) == _decode_rule(*r[:5]), r
    # the decode sweep's shape takes the decode kernel, the skinny batch shapes do not
    assert _decode_rule(1, 4096, 4096, 128, 152) and not _decode_rule(16, 14336, 4096, 64, 152)
