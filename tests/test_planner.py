"""Host-side checks of the skinny kernel's planner (no GPU needed).

tests/planner_check.cu compiles the planner (bit_weight_quantized_gb300/csrc/
gemv.cu) into a host program that prints each plan.  The plans must cover
every row and every K chunk, keep the padded pitch that makes the MMA quads'
reads conflict-free, lay out shared memory without overlap inside the per-CTA
limit, and fit the decode shapes in half an SM (two CTAs per SM, so that
consecutive calls overlap).

tests/decode_route_check.cu does the same for the decode kernel's shape rule
and launch plan (bit_weight_quantized_gb300/csrc/decode.cu, decode_plan), checked against
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
DECODE_FIELDS = ("grid", "rows_base", "rows_rem", "max_rows", "warps", "kseg", "nseg", "seg_bytes", "span", "pitch",
                 "slot_bytes", "slots", "x_pitch", "off_x", "off_xsum", "off_sc", "off_zo", "off_red",
                 "off_bar", "smem")
SMEM_PAIR, SMEM_OPTIN = 115712, 232448   # GB300: half an SM's shared memory per CTA, and the opt-in limit


_DECODE_EXE = {}


def decode_plans(shapes, tmp_dir):
    """Runs tests/decode_route_check.cu on (M, N, K, G, bits, zeros, sms, pair, optin
    [, tile16]) tuples; returns None (skinny kernel) or a dict of the DecodePlan per
    shape."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = _DECODE_EXE.get("path")
    if exe is None:   # compiled once per test process (the kernels make it slow to build)
        exe = os.path.join(str(tmp_dir), "decode_route_check")
        subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                        "--expt-relaxed-constexpr", "-o", exe, os.path.join(HERE, "decode_route_check.cu")],
                       check=True, capture_output=True)
        _DECODE_EXE["path"] = exe
    stdin = "".join(" ".join(map(str, sh[:9])) + f" {sh[9] if len(sh) > 9 else 0}\n" for sh in shapes)
    out = subprocess.run([exe], input=stdin, capture_output=True, text=True, check=True).stdout
    res = []
    for line, sh in zip(out.splitlines(), shapes):
        v = list(map(int, line.split()))
        assert tuple(v[:9]) == tuple(sh[:9])
        res.append(dict(zip(DECODE_FIELDS, v[10:])) if v[9] else None)
    assert len(res) == len(shapes)
    return res


def _decode_shapes():
    s = []
    for sms in (152, 148, 4):
        for b in range(1, 9):
            for M in (1, 3, 8, 9, 16, 17):
                for (N, K, G, z) in [(4096, 4096, 128, 0), (11008, 4096, 64, 1), (14336, 4096, 64, 1),
                                     (37, 512, 64, 1), (300, 1024, 128, 0), (4000, 512, 64, 0),
                                     (1, 2048, 128, 0), (4865, 1024, 128, 1), (20000, 65536, 128, 0),
                                     (150, 1536, 128, 1), (64, 1000, 64, 0), (64, 768, 128, 0),
                                     (64, 1024, 32, 0)]:
                    s.append((M, N, K, G, b, z, sms, SMEM_PAIR, SMEM_OPTIN))
    return s


@pytest.fixture(scope="module")
def dplans(tmp_path_factory):
    shapes = _decode_shapes()
    return list(zip(shapes, decode_plans(shapes, tmp_path_factory.mktemp("decode"))))


def test_decode_route_rule(dplans):
    # the shapes the kernel may take: 1 <= M <= 16, groups of 64 / 128, K a positive
    # multiple of 8 groups; the rest go to the skinny kernel
    for (M, N, K, G, b, z, sms, pair, optin), pl in dplans:
        eligible = 1 <= M <= 16 and G in (64, 128) and K >= 8 * G and K % (8 * G) == 0
        if not eligible:
            assert pl is None, (M, N, K, G, b)
    plan = {sh[:6] + (sh[6],): pl for sh, pl in dplans}
    for b in range(1, 9):
        # the decode sweep and the skinny batched-decode shapes take the staged kernel
        assert plan[(1, 4096, 4096, 128, b, 0, 152)] is not None
        for M in (3, 8, 9, 16):
            assert plan[(M, 14336, 4096, 64, b, 1, 152)] is not None
            assert plan[(M, 11008, 4096, 64, b, 1, 152)] is not None


def test_decode_plan_layout(dplans):
    resid = {1: 16, 2: 16, 3: 16, 4: 32, 5: 16, 6: 16, 7: 16, 8: 64}
    for (M, N, K, G, b, z, sms, pair, optin), pl in dplans:
        if pl is None:
            continue
        key = (M, N, K, G, b, z, sms)
        assert pl["grid"] == min(N, sms), key
        assert pl["grid"] * pl["rows_base"] + pl["rows_rem"] == N and pl["rows_rem"] < pl["grid"], key
        assert pl["max_rows"] == pl["rows_base"] + (pl["rows_rem"] > 0), key
        # 8 warps; warp w owns group w of every segment
        assert pl["warps"] == 8, key
        assert pl["kseg"] == 8 * G and pl["nseg"] * pl["kseg"] == K, key
        assert pl["seg_bytes"] == pl["kseg"] * b // 8 and pl["seg_bytes"] % 16 == 0, key
        # a slot holds whole rows (every row block at once) or one segment
        assert pl["span"] in (1, pl["nseg"]), key
        chunk = pl["span"] * pl["seg_bytes"]
        assert pl["pitch"] >= chunk and pl["pitch"] % 16 == 0, key
        assert pl["pitch"] % 128 == resid[b], key
        slot_rows = min(32, pl["max_rows"])
        if pl["pitch"] <= 2048:
            # slots that one tensor-map box fills start on 128 bytes
            assert pl["slot_bytes"] == _ceil(slot_rows * pl["pitch"], 128) * 128, key
        else:
            assert pl["slot_bytes"] == slot_rows * pl["pitch"], key
        total = _ceil(pl["max_rows"], 32) * (pl["nseg"] // pl["span"])
        assert 1 <= pl["slots"] <= min(total, 16), key
        assert pl["slots"] == total or pl["slots"] >= 2, key
        if pl["span"] == pl["nseg"] and pl["nseg"] > 1:
            assert pl["slots"] == total, key
        # regions in order, aligned, without overlap, inside the budget
        assert pl["slots"] * pl["slot_bytes"] <= pl["off_x"] and pl["off_x"] % 16 == 0, key
        assert pl["x_pitch"] == K // pl["warps"] * 2 + 16, key
        assert pl["off_x"] + pl["warps"] * M * pl["x_pitch"] <= pl["off_xsum"], key
        assert pl["off_xsum"] + pl["warps"] * M * pl["nseg"] * 8 <= pl["off_sc"], key   # (X, C) pairs
        ng = K // G
        assert pl["off_sc"] + pl["max_rows"] * ng * 2 <= pl["off_zo"], key
        assert pl["off_zo"] + (pl["max_rows"] * ng * 2 if z else 0) <= pl["off_red"], key
        assert pl["off_red"] + pl["warps"] * 32 * M * 4 <= pl["off_bar"] and pl["off_bar"] % 8 == 0, key
        assert pl["off_bar"] + 2 * pl["slots"] * 8 + 4 <= pl["smem"] <= optin, key


def test_decode_sweep_keeps_two_ctas_per_sm_and_preloads(dplans):
    # the decode sweep fits two CTAs per SM (one call computing while the next
    # one's weights stream in); up to b = 7 a CTA's whole weight share is in
    # flight before its dependency wait, at b = 8 three quarters
    for (M, N, K, G, b, z, sms, pair, optin), pl in dplans:
        if (M, N, K, G, z, sms) == (1, 4096, 4096, 128, 0, 152):
            assert pl["smem"] <= SMEM_PAIR, b
            if b <= 7:   # one bulk copy per row, the whole of K
                assert pl["span"] == pl["nseg"] and pl["slots"] == 1, b
            else:
                assert pl["span"] == 1 and pl["slots"] * 4 >= pl["nseg"] * 3, b


def test_decode_plan_tile16_layout(tmp_path_factory):
    # the fragment-ordered layout: CTAs own whole 16-row tiles, slots hold two
    # dense tiles, everything else as for the canonical layout
    shapes = [(M, N, K, G, b, z, sms, SMEM_PAIR, SMEM_OPTIN, 1)
              for sms in (152, 4) for b in (1, 3, 4, 8) for M in (1, 9, 16)
              for (N, K, G, z) in [(4096, 4096, 128, 0), (14336, 4096, 64, 1), (37, 1024, 128, 1), (8, 2048, 64, 0)]]
    plans = decode_plans(shapes, tmp_path_factory.mktemp("tile"))
    for sh, pl in zip(shapes, plans):
        M, N, K, G, b, z, sms = sh[:7]
        if pl is None:
            continue
        tiles = -(-N // 16)
        assert pl["grid"] == min(tiles, sms), sh
        assert pl["grid"] * pl["rows_base"] + pl["rows_rem"] == tiles, sh
        assert pl["max_rows"] == min(16 * (pl["rows_base"] + (pl["rows_rem"] > 0)), N), sh
        assert pl["pitch"] == 0 and pl["slot_bytes"] == 32 * pl["span"] * pl["seg_bytes"], sh
        assert pl["slots"] * pl["slot_bytes"] <= pl["off_x"] and pl["smem"] <= SMEM_OPTIN, sh
    sweep = {sh[4]: pl for sh, pl in zip(shapes, plans) if sh[:4] == (1, 4096, 4096, 128) and sh[6] == 152}
    for b in (1, 3, 4):
        assert sweep[b]["span"] == sweep[b]["nseg"] and sweep[b]["smem"] <= SMEM_PAIR, b


def test_stage_tensor_box_fits(plans):
    # where the skinny kernel lands a stage with one tensor copy (pitch <= 2048
    # bytes in 16-byte units, 16-byte rows and segments: skinny_set_tma), the box
    # of rb rows x pitch bytes stays inside its stage, and the stages start on
    # 128 bytes (the kernel checks this too and falls back to bulk copies)
    n = 0
    for p in plans:
        if p["st"] != 0:
            continue
        row_bytes = p["K"] * p["bits"] // 8
        if p["pitch"] % 16 or p["pitch"] > 2048 or row_bytes % 16 or p["seg_bytes"] % 16:
            continue
        n += 1
        key = (p["M"], p["N"], p["K"], p["bits"], p["group"])
        assert p["rb"] * p["pitch"] <= p["stage_bytes"], key
        assert p["off_ring"] % 128 == 0 and p["stage_bytes"] % 128 == 0, key
        assert p["off_ring"] + p["ring"] * p["stage_bytes"] <= p["smem"], key
    assert n > 0
