"""Host emulation of the decode kernel's bit-level steps (no GPU needed).

bit_weight_quantized_gb300/csrc/decode.cu turns each thread's packed words
into fp16 MMA operands with funnel shifts, byte permutes and LOP3s, and
permutes the MMA's k order so that the B fragment is one contiguous slice
of x.  These tests restate those integer operations in Python, exactly as
the kernel performs them, and check the invariants the kernel relies on:
- every extracted fp16 half is exactly 2^E + q for its code q;
- a thread's words for one row and 64-code block lie inside that block, and
  the 8- / 16-byte loads at b = 4 / 8 are aligned;
- the permuted k order, placed into the m16n8k16 fragment layout, gives the
  same product as the plain sum over the block's codes.
"""
import numpy as np
import pytest

from synthetic import SplitMix64

M32 = 0xFFFFFFFF


# ---- the kernel's integer operations, restated ------------------------------------
def funnelshift_r(lo, hi, s):
    return (((hi << 32) | lo) >> (s & 31)) & M32


def prmt(a, b, sel):
    by = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    return sum(by[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def lop3_and_or(a, mask, bits):
    return (a & mask) | bits


def dec_words(b):
    return (b + 1) // 2


def dec_exp(b):
    return 10 if b in (4, 8) else b


def dec_pair(b, win, c):
    """fp16 pair of codes c, c + 1 of a thread's 16 codes (code 0 at bit 0 of win[0])."""
    if b == 8:
        return prmt(win[c >> 2], 0x64646464, 0x4342 if c & 2 else 0x4140)
    if b == 4:
        w = win[c >> 3]
        byte = (c & 7) >> 1
        return lop3_and_or(prmt(w, w >> 4, byte | ((4 + byte) << 8)), 0x000F000F, 0x64006400)
    sh = c * b - (10 - b)
    u = (win[0] << (-sh)) & M32 if sh < 0 else funnelshift_r(win[sh >> 5], win[(sh >> 5) + 1], sh & 31)
    mask = ((1 << b) - 1) << (10 - b)
    magic = (b + 15) << 10
    lo = lop3_and_or(u, mask, magic | (magic << 16))
    return lop3_and_or((u << (16 - b)) & M32, (mask << 16) & M32, lo)


def thread_window(b, words, t):
    """The thread's shifted window: words read at its first word, shifted by its
    bit offset (odd widths only), plus one zero word."""
    nw = dec_words(b)
    o = 16 * (t & 1) if b & 1 else 0
    first = (16 * b * t) // 32
    raw = [int(words[first + k]) for k in range(nw)]
    win = [funnelshift_r(raw[k], raw[k + 1] if k + 1 < nw else 0, o) if b & 1 else raw[k]
           for k in range(nw)]
    return win + [0]


def pack_block(codes, b):
    """LSB-first bitstream of one 64-code block as 32-bit words (2b words)."""
    bits = ((codes[:, None].astype(np.int64) >> np.arange(b)) & 1).reshape(-1).astype(np.uint8)
    return np.packbits(bits, bitorder="little").view("<u4").astype(np.int64)


def half(bits16):
    return float(np.array([bits16 & 0xFFFF], dtype=np.uint16).view(np.float16)[0])


# ---- tests ------------------------------------------------------------------------
@pytest.mark.parametrize("b", range(1, 9))
def test_pairs_are_exactly_pow2_plus_code(b):
    st = SplitMix64(100 + b)
    for trial in range(24):
        codes = st.uniform_bits(64, b).astype(np.int64)
        if trial == 0:
            codes[:] = (1 << b) - 1          # all ones
        elif trial == 1:
            codes[:] = 0
        words = pack_block(codes, b)
        assert len(words) == 2 * b
        for t in range(4):
            win = thread_window(b, words, t)
            for c in range(0, 16, 2):
                pr = dec_pair(b, win, c)
                assert half(pr) == 2.0 ** dec_exp(b) + codes[16 * t + c], (b, t, c)
                assert half(pr >> 16) == 2.0 ** dec_exp(b) + codes[16 * t + c + 1], (b, t, c)


@pytest.mark.parametrize("b", range(1, 9))
@pytest.mark.parametrize("K", [512, 1024, 4096, 11008 // 512 * 512, 65536])
def test_thread_words_stay_in_block_and_vector_loads_align(b, K):
    row_words = K * b // 32
    kw = K // 8
    nw = dec_words(b)
    for row in (0, 1, 7):
        for warp in range(8):
            k0w = warp * kw
            for j in range(kw // 64):
                block_lo = (k0w * b + 64 * b * j) // 32
                block_hi = (k0w * b + 64 * b * (j + 1)) // 32
                for t in range(4):
                    first = (k0w * b + 16 * b * t) // 32 + 2 * b * j
                    assert block_lo <= first and first + nw <= block_hi
                    # the last code's bits lie inside the words read
                    o = (16 * b * t) % 32
                    assert o + 16 * b <= 32 * nw
                    if b in (4, 8):
                        # byte address relative to a 16-byte aligned base
                        assert ((row * row_words + first) * 4) % (4 * nw) == 0


@pytest.mark.parametrize("b", range(1, 9))
def test_permuted_k_order_gives_the_plain_dot_product(b):
    """One warp, one 64-code block, two 16-row tiles, 8 tokens: the fragments
    each thread supplies, placed by the m16n8k16 layout, multiply to
    sum_k (2^E + q[r][k]) x[m][k] for every row r and token m."""
    st = SplitMix64(7 * b)
    rows = 32
    codes = st.uniform_bits(rows * 64, b).reshape(rows, 64).astype(np.int64)
    x = (st.normal(8 * 64).reshape(8, 64)).astype(np.float16).astype(np.float64)
    words = [pack_block(codes[r], b) for r in range(rows)]
    D = np.zeros((rows, 8))
    for s in range(4):
        for i in range(2):
            A = np.zeros((16, 16))
            Bm = np.zeros((16, 8))
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                wins = [thread_window(b, words[16 * i + 8 * h + g], t) for h in range(2)]
                regs = [dec_pair(b, wins[0], 4 * s), dec_pair(b, wins[1], 4 * s),
                        dec_pair(b, wins[0], 4 * s + 2), dec_pair(b, wins[1], 4 * s + 2)]
                places = [(g, 2 * t), (g + 8, 2 * t), (g, 2 * t + 8), (g + 8, 2 * t + 8)]
                for r, (row, k) in zip(regs, places):
                    A[row, k], A[row, k + 1] = half(r), half(r >> 16)
                base = 16 * t + 4 * s   # the B fragment: x[16t + 4s .. 16t + 4s + 3] of token g
                Bm[2 * t, g], Bm[2 * t + 1, g] = x[g, base], x[g, base + 1]
                Bm[2 * t + 8, g], Bm[2 * t + 9, g] = x[g, base + 2], x[g, base + 3]
            D[16 * i:16 * i + 16] += A @ Bm
    ref = (2.0 ** dec_exp(b) + codes.astype(np.float64)) @ x.T
    np.testing.assert_allclose(D, ref, rtol=0, atol=1e-9 * np.abs(ref).max())


# ---- the staged kernel end to end: placement in shared memory, reads, fold ----------
def _f16_bits_of_int(v):
    e = v.bit_length() - 1
    return ((e + 15) << 10) | ((v << (10 - e)) & 0x3FF)


def _plan_pairs(b, run):
    """The 8 fp16 pairs of a thread's normalized 16-code run (words, code 0 at
    bit 0), through the generated plan exactly as the kernel builds them:
    [(2^E_lo + q_lo, 2^E_hi + q_hi)] in pair order, as exact fp16 values."""
    from tests.test_unpack_plans import PLANS, _window
    if b == 8:
        out = []
        for i in range(8):
            v = prmt(run[i >> 1], 0x64646464, 0x4342 if i & 1 else 0x4140)
            out.append((half(v), half(v >> 16)))
        return out
    P = PLANS[(b, 16)]
    wins = [_window(run, P, u) for u in range(P["kWindows"])]
    out = []
    for i in range(8):
        v = (wins[P["win"][i]] & P["mask"][i]) | P["magic"][i]
        out.append((half(v), half(v >> 16)))
    return out


def _slot_codes(b):
    """code_of_slot: the run code whose activation sits in fragment slot s."""
    from tests.test_unpack_plans import PLANS
    if b == 8:
        return list(range(16))
    P = PLANS[(b, 16)]
    out = []
    for s in range(16):
        i = 2 * (s >> 2) + ((s >> 1) & 1)
        out.append(P["hi"][i] if s & 1 else P["lo"][i])
    return out


def _code_exps(b):
    """exp_of_code: E of each run code (its operand is 2^E + q)."""
    from tests.test_unpack_plans import PLANS
    if b == 8:
        return [10] * 16
    P = PLANS[(b, 16)]
    e = [None] * 16
    for i in range(8):
        e[P["lo"][i]] = P["elo"][i]
        e[P["hi"][i]] = P["ehi"][i]
    return e


def _emulate_staged(prob, packed, plan, tile16=False, ix_sa=None, acc_out=None):
    """y of the staged decode kernel, emulated from its plan: bulk copies place each
    row's chunk in a ring slot at the plan's pitch; each warp stages its group of
    every segment in fragment (slot) order and forms X and C per group; every lane
    reads its run words and activation fragments back through the kernel's
    address formulas (asserting each read stays in its region), extracts its code
    pairs 2^E + q with the generated plan, and the MMA order follows the pairs.
    Products and sums are exact (fp64 over exact fp16 values); the group fold is
    s (acc - C - z X).  With ix_sa (the per-token scales) it emulates the
    exact-integer mode instead: prob.x holds the int8 activations as fp16, the
    words of the signed stream are XORed to offset binary before extraction and
    each operand loses its 2^E, C = 0, and the accumulators acc - z X go to
    acc_out[m][n][g]; y is scaled by ix_sa[m]."""
    ix = ix_sa is not None
    b, M, N, K, G = prob.bits, prob.M, prob.N, prob.K, prob.group
    ng = K // G
    nw = dec_words(b)
    NB = G // 64
    row_bytes = K * b // 8
    W, kseg, nseg, S = plan["warps"], plan["kseg"], plan["nseg"], plan["slots"]
    assert W == 8 and kseg == 8 * G
    pitch, slot_bytes, xp = plan["pitch"], plan["slot_bytes"], plan["x_pitch"]
    slot_rows = min(32, plan["max_rows"])
    xf = prob.x.astype(np.float64)
    xbits = prob.x.view(np.uint16)
    scb = prob.scales.view(np.uint16)
    slot_code = _slot_codes(b)
    slots, exps = slot_code, _code_exps(b)
    y = np.zeros((M, N))
    for cta in range(plan["grid"]):
        u0 = cta * plan["rows_base"] + min(cta, plan["rows_rem"])
        nu = plan["rows_base"] + (1 if cta < plan["rows_rem"] else 0)
        r0 = 16 * u0 if tile16 else u0
        nrows = min(16 * nu, N - r0) if tile16 else nu
        sm = np.zeros(plan["smem"], dtype=np.uint8)
        # scales / zeros of the CTA's rows, transposed to [group][row]
        sc = np.zeros(ng * nrows, dtype=np.uint16)
        zo = np.zeros(ng * nrows) if prob.zeros is not None else None
        for e in range(nrows * ng):
            row, gi = divmod(e, ng)
            sc[gi * nrows + row] = scb[r0 + row, gi]
            if zo is not None:
                zo[gi * nrows + row] = float(prob.zeros[r0 + row, gi])
        assert nrows * ng * 2 <= plan["off_zo"] - plan["off_sc"]
        # activations: warp w's group of every segment, every token, in slot order;
        # the group sums X[w][m][j] and offsets C[w][m][j] = sum 2^E x
        xend = plan["off_x"] + W * M * xp
        X = np.zeros((W, M, nseg))
        C = np.zeros((W, M, nseg))
        pw = 2.0 ** np.array(_code_exps(b), dtype=np.float64)
        for w in range(W):
            for m in range(M):
                for j in range(nseg):
                    for bb in range(NB):
                        for tq in range(4):
                            dst = plan["off_x"] + w * M * xp + m * xp + ((j * NB + bb) * 64 + 16 * tq) * 2
                            src = j * kseg + 64 * (w * NB + bb) + 16 * tq
                            assert plan["off_x"] <= dst and dst + 32 <= xend and src + 16 <= K
                            run = xbits[m, src:src + 16]
                            sm[dst:dst + 32] = run[slot_code].view(np.uint8)
                            X[w, m, j] += xf[m, src:src + 16].sum()
                            if not ix:   # the integer mode's operands carry no offset
                                C[w, m, j] += (pw * xf[m, src:src + 16]).sum()
        assert plan["off_xsum"] + W * M * nseg * 8 <= plan["off_sc"]   # (X, C) fp32 pairs
        nrb = -(-nrows // 32)
        span = plan["span"]
        chunk = span * plan["seg_bytes"]
        # the rule of decode_tma_fits (decode.h): one tensor-map box of a slot's
        # rows per chunk where the pitch is at most 2048 bytes
        box_rows = min(32, plan["max_rows"])
        tma = (not tile16 and pitch % 16 == 0 and 0 < pitch <= 2048 and row_bytes % 16 == 0
               and chunk % 16 == 0)
        for rb in range(nrb):
            rr = 32 * rb
            cnt = min(32, nrows - rr)
            tot = np.zeros((W, 32, M))
            for j in range(nseg):
                c, jj = divmod(j, span)
                i = rb * (nseg // span) + c
                slot = i % S
                base = slot * slot_bytes
                if jj == 0 and tile16:   # the chunk's bulk copies: one per 16-row tile
                    for ti in range(-(-cnt // 16)):
                        dst = base + ti * 16 * chunk
                        assert dst + 16 * chunk <= base + slot_bytes <= plan["off_x"]
                        src = (r0 + rr) * row_bytes + c * 16 * chunk + ti * 16 * row_bytes
                        assert src + 16 * chunk <= packed.size
                        sm[dst:dst + 16 * chunk] = packed.reshape(-1)[src:src + 16 * chunk]
                elif jj == 0 and tma:   # one tensor-map box: a slot's rows x pitch bytes (zeros outside)
                    flat = packed.reshape(-1)
                    assert base % 128 == 0 and (c * chunk) % 16 == 0 and box_rows >= cnt
                    assert base + box_rows * pitch <= base + slot_bytes <= plan["off_x"]
                    for r in range(box_rows):
                        row = r0 + rr + r
                        n = max(0, min(pitch, row_bytes - c * chunk)) if row < N else 0
                        src = row * row_bytes + c * chunk
                        sm[base + r * pitch:base + (r + 1) * pitch] = 0
                        sm[base + r * pitch:base + r * pitch + n] = flat[src:src + n]
                elif jj == 0:   # the chunk's bulk copies: one per row
                    for r in range(cnt):
                        dst = base + r * pitch
                        assert dst + chunk <= base + slot_rows * pitch <= plan["off_x"]
                        src = (r0 + rr + r) * row_bytes + c * chunk
                        sm[dst:dst + chunk] = packed.reshape(-1)[src:src + chunk]
                for w in range(W):
                    gidx = j * W + w
                    acc = np.zeros((32, M))
                    for bb in range(NB):
                        A = np.zeros((32, 16 * 4))    # [row][16 t + slot] = q of the code in that slot
                        for g in range(8):
                            for t in range(4):
                                first_b = (16 * b * t) // 32 * 4
                                o = 16 * (t & 1) if b & 1 else 0
                                for i2 in range(2):
                                    for h in range(2):
                                        row = 16 * i2 + 8 * h + g
                                        lr = min(row, cnt - 1)
                                        kblock = jj * (kseg // 64) + w * NB + bb
                                        if tile16:   # the padding rows of a tile are real zero codes
                                            a = (base + i2 * 16 * chunk + kblock * 128 * b + ((8 * h + g) * 4 + t) * 2 * b
                                                 - (2 if (b & 1) and (t & 1) else 0))
                                            assert base <= a and a + 4 * nw <= base + slot_bytes
                                            if row >= cnt:
                                                continue
                                        else:
                                            a = base + lr * pitch + kblock * 8 * b + first_b
                                            assert base <= a and a + 4 * nw <= base + lr * pitch + (jj + 1) * plan["seg_bytes"]
                                        if b == 4:
                                            assert a % 8 == 0
                                        if b == 8:
                                            assert a % 16 == 0
                                        raw = [int(v) for v in sm[a:a + 4 * nw].view("<u4")]
                                        if ix:   # two's complement -> offset binary
                                            raw = [v ^ (0x88888888 if b == 4 else 0x80808080) for v in raw]
                                        run = [funnelshift_r(raw[k], raw[k + 1] if k + 1 < nw else 0, o)
                                               if b & 1 else raw[k] for k in range(nw)]
                                        for pi, (qlo, qhi) in enumerate(_plan_pairs(b, run)):
                                            if ix:   # the plan's offsets come off: the codes themselves
                                                qlo -= 2.0 ** exps[slots[2 * pi]]
                                                qhi -= 2.0 ** exps[slots[2 * pi + 1]]
                                            jp, hp = divmod(pi, 2)
                                            A[row, 16 * t + 4 * jp + 2 * hp] = qlo
                                            A[row, 16 * t + 4 * jp + 2 * hp + 1] = qhi
                        Xf = np.zeros((64, M))
                        for m in range(M):
                            for t in range(4):
                                a = plan["off_x"] + w * M * xp + m * xp + ((j * NB + bb) * 64 + 16 * t) * 2
                                assert a + 32 <= xend
                                Xf[16 * t:16 * t + 16, m] = sm[a:a + 32].view(np.float16).astype(np.float64)
                        acc += A @ Xf
                    for row in range(32):
                        lr = min(row, cnt - 1)
                        e = gidx * nrows + rr + lr
                        s = float(np.array([sc[e]], dtype=np.uint16).view(np.float16)[0])
                        z = zo[e] if zo is not None else float(prob.zero_const)
                        tot[w, row] += s * (acc[row] - C[w, :, j] - z * X[w, :, j])
                        if ix and acc_out is not None and row < cnt:
                            acc_out[:, r0 + rr + row, gidx] = acc[row] - z * X[w, :, j]
            y[:, r0 + rr:r0 + rr + cnt] = tot.sum(axis=0)[:cnt].T
    if ix:
        y = y * np.asarray(ix_sa, dtype=np.float64)[:, None]
    return y


@pytest.mark.parametrize("b,M,N,K,G,zm,sms", [
    (4, 1, 40, 1024, 128, "half", 4), (3, 3, 75, 1024, 64, "group", 2),
    (8, 2, 37, 2048, 128, "group", 1), (1, 9, 33, 512, 64, "const8", 1),
    (7, 2, 66, 1024, 128, "half", 2), (5, 1, 8, 2048, 64, "group", 4),
    (6, 16, 20, 1024, 128, "half", 1), (2, 4, 19, 1024, 64, "group", 1)])
def test_staged_kernel_emulation_matches_oracle(b, M, N, K, G, zm, sms, tmp_path):
    import oracle
    import synthetic
    from tests.test_planner import SMEM_OPTIN, SMEM_PAIR, decode_plans
    prob = synthetic.make_qmm(M, N, K, b, G, zero_mode=zm, seed=b + 10 * M)
    # a small SM count gives several row blocks per CTA and rows past 32
    plan = decode_plans([(M, N, K, G, b, 1 if prob.zeros is not None else 0, sms, SMEM_PAIR, SMEM_OPTIN)],
                        tmp_path)[0]
    assert plan is not None
    packed, _ = oracle.pack(prob.codes, b)
    y = _emulate_staged(prob, packed, plan)
    ref = oracle.solve_qmm(prob)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-9 * max(1.0, np.abs(ref).max()))


@pytest.mark.parametrize("b,M,N,K,G,zm,sms", [
    (4, 1, 40, 1024, 128, "half", 2), (3, 3, 75, 1024, 64, "group", 2), (8, 2, 37, 2048, 128, "group", 1),
    (7, 9, 20, 512, 64, "const8", 1), (5, 1, 8, 2048, 64, "group", 4)])
def test_staged_kernel_emulation_tile16(b, M, N, K, G, zm, sms, tmp_path):
    # the fragment-ordered layout (written by the oracle's tile16): one bulk copy
    # per tile, runs read at their tile16 offsets
    import oracle
    import synthetic
    from tests.test_planner import SMEM_OPTIN, SMEM_PAIR, decode_plans
    prob = synthetic.make_qmm(M, N, K, b, G, zero_mode=zm, seed=b + 7 * M)
    plan = decode_plans([(M, N, K, G, b, 1 if prob.zeros is not None else 0, sms, SMEM_PAIR, SMEM_OPTIN, 1)],
                        tmp_path)[0]
    assert plan is not None
    y = _emulate_staged(prob, oracle.tile16(prob.codes, b), plan, tile16=True)
    ref = oracle.solve_qmm(prob)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-9 * max(1.0, np.abs(ref).max()))


def test_staged_kernel_emulation_small_ring(tmp_path):
    # a budget that leaves two slots for eight segments: the ring is reused
    import oracle
    import synthetic
    from tests.test_planner import decode_plans
    prob = synthetic.make_qmm(2, 40, 4096, 8, 128, zero_mode="half", seed=3)
    plan = decode_plans([(2, 40, 4096, 128, 8, 0, 1, 95000, 95000)], tmp_path)[0]
    assert plan is not None and plan["slots"] < 2 * plan["nseg"]
    y = _emulate_staged(prob, oracle.pack(prob.codes, 8)[0], plan)
    ref = oracle.solve_qmm(prob)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-9 * np.abs(ref).max())


@pytest.mark.parametrize("b,M,N,K,G,zm,budget", [
    (6, 4, 40, 4096, 64, "group", 95000), (4, 2, 25, 8192, 128, "half", 75000),
    (8, 1, 37, 2048, 64, "group", 60000), (3, 16, 70, 4096, 64, "const8", 196000)])
def test_staged_kernel_emulation_tma_boxes(b, M, N, K, G, zm, budget, tmp_path):
    # one-segment ring slots landed by one tensor-map box each (the canonical
    # layout's rule in decode.h; the other emulation cases take it too where the
    # pitch allows): each box stays inside its slot, rows past N and bytes past a
    # row's end arrive as zeros, and the result is the oracle's
    import oracle
    import synthetic
    from tests.test_planner import decode_plans
    prob = synthetic.make_qmm(M, N, K, b, G, zero_mode=zm, seed=b + 5 * M)
    plan = decode_plans([(M, N, K, G, b, 1 if prob.zeros is not None else 0, 1, budget, budget)],
                        tmp_path)[0]
    assert plan is not None and plan["span"] == 1 and plan["pitch"] <= 2048
    y = _emulate_staged(prob, oracle.pack(prob.codes, b)[0], plan)
    ref = oracle.solve_qmm(prob)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-9 * max(1.0, np.abs(ref).max()))


@pytest.mark.parametrize("b,M,N,K,G,sms", [
    (4, 1, 40, 1024, 128, 4), (4, 3, 75, 1024, 64, 2), (4, 8, 37, 2048, 128, 1), (4, 5, 20, 512, 64, 1),
    (8, 1, 33, 1024, 128, 2), (8, 4, 19, 512, 64, 1), (8, 2, 66, 2048, 64, 4)])
def test_staged_kernel_emulation_integer_mode(b, M, N, K, G, sms, tmp_path):
    # the exact-integer mode of qmm_w4a8 / qmm_w8a8 (int8 activations, signed
    # codes as offset binary, the plan's offsets taken off each operand): its
    # accumulators equal the oracle's integers and its output the oracle's y
    from types import SimpleNamespace
    import oracle
    import synthetic
    from tests.test_planner import SMEM_OPTIN, SMEM_PAIR, decode_plans
    if b == 4:
        prob = synthetic.make_w4a8(M, N, K, G, seed=M * 11 + N)
        codes = prob.w4
        y_ref, acc_ref, ov = oracle.solve_w4a8(prob)
    else:
        prob = synthetic.make_w8a8(M, N, K, G, seed=M * 13 + N)
        codes = prob.w8.view(np.uint8)
        y_ref, acc_ref, ov = oracle.solve_w8a8(prob)
    assert not ov
    view = SimpleNamespace(bits=b, M=M, N=N, K=K, group=G, x=prob.xq.astype(np.float16), scales=prob.ws,
                           zeros=None, zero_const=1 << (b - 1))
    plan = decode_plans([(M, N, K, G, b, 0, sms, SMEM_PAIR, SMEM_OPTIN)], tmp_path)[0]
    assert plan is not None
    acc = np.zeros((M, N, K // G))
    y = _emulate_staged(view, oracle.pack(codes, b)[0], plan, ix_sa=prob.sa.astype(np.float64), acc_out=acc)
    np.testing.assert_array_equal(acc, acc_ref.astype(np.float64))
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())


def _float_pair_bits(word, q, b, e, m):
    """Emulates the decode kernel's float extraction of pair q of a 32-bit word
    (b = 4: nibbles 2j, 2j + 1 of the word, j = q % 4; b = 8: bytes 2(q % 2),
    2(q % 2) + 1): byte permute, masked field shifted to the top of the fp16
    exponent/mantissa fields, sign to bit 15 of each half."""
    def prmt(a, bb, sel):
        src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(bb >> (8 * i)) & 0xFF for i in range(4)]
        return sum(src[(sel >> (4 * k)) & 7] << (8 * k) for k in range(4))
    if b == 4:
        j = q & 3
        t = prmt(word, word >> 4, j | ((4 + j) << 8))
    else:
        b0 = 2 * (q & 1)
        t = prmt(word, 0, b0 | (4 << 4) | ((b0 + 1) << 8) | (4 << 12))
    mask = ((1 << (e + m)) - 1) * 0x00010001
    em = ((t & mask) << (10 - m)) & 0xFFFFFFFF
    sg = (t << (15 - e - m)) & 0x80008000
    return em | sg


def _float_pair_bits_any(run, q, b, e, m):
    """The extraction at widths other than 4 and 8: run = the 16-code run as an
    integer (code k at bit b k); codes 2q and 2q + 1 are each shifted to bit 0 of
    a 32-bit word (the following codes above them) and the low halves joined,
    then masked and shifted as at b = 4, 8."""
    nbits = 32 * ((b + 1) // 2)
    def at0(k):
        return (run >> (b * k)) & 0xFFFFFFFF if b * k < nbits else 0
    t = (at0(2 * q) & 0xFFFF) | ((at0(2 * q + 1) & 0xFFFF) << 16)
    mask = ((1 << (e + m)) - 1) * 0x00010001
    em = ((t & mask) << (10 - m)) & 0xFFFFFFFF
    sg = (t << (15 - e - m)) & 0x80008000
    return em | sg


@pytest.mark.parametrize("b,e", [(2, 1), (3, 1), (3, 2), (5, 2), (5, 4), (6, 3), (7, 3), (7, 4)])
def test_float_code_extraction_any_width_is_exact(b, e):
    import oracle
    m = b - 1 - e
    bias = (1 << (e - 1)) - 1
    st = np.random.default_rng(b * 10 + e)
    for q in range(8):
        for c in range(1 << b):
            for c2 in (0, (1 << b) - 1, c ^ 1):
                codes = [int(v) for v in st.integers(0, 1 << b, 16)]
                codes[2 * q], codes[2 * q + 1] = c, c2
                run = sum(v << (b * k) for k, v in enumerate(codes))
                bits = _float_pair_bits_any(run, q, b, e, m)
                lo = np.array([bits & 0xFFFF], dtype=np.uint16).view(np.float16)[0]
                hi = np.array([bits >> 16], dtype=np.uint16).view(np.float16)[0]
                assert float(lo) == oracle.float_value(c, e, m) * 2.0 ** (bias - 15)
                assert float(hi) == oracle.float_value(c2, e, m) * 2.0 ** (bias - 15)


@pytest.mark.parametrize("b,e", [(4, 1), (4, 2), (4, 3), (8, 1), (8, 2), (8, 3), (8, 4)])
def test_float_code_extraction_is_exact(b, e):
    # every code of the split through the extraction: fp16 value = code value * 2^(bias - 15).
    # (e = 5 is left to the FFMA kernel: its top exponent field would read as inf in fp16)
    import oracle
    m = b - 1 - e
    bias = (1 << (e - 1)) - 1
    for q in range(8 if b == 4 else 2):
        for c in range(1 << b):
            for c2 in (0, (1 << b) - 1, c ^ 1):
                if b == 4:   # code c at nibble 2j, c2 at 2j + 1 of a word, other nibbles noise
                    j = q & 3
                    word = 0x9A5C3E71 & ~(0xFF << (8 * j)) | (c << (8 * j)) | (c2 << (8 * j + 4))
                else:        # code c at byte 2(q % 2), c2 at the next byte
                    b0 = 2 * (q & 1)
                    word = 0xB4D27E19 & ~(0xFFFF << (8 * b0)) | (c << (8 * b0)) | (c2 << (8 * b0 + 8))
                bits = _float_pair_bits(word, q, b, e, m)
                lo = np.array([bits & 0xFFFF], dtype=np.uint16).view(np.float16)[0]
                hi = np.array([bits >> 16], dtype=np.uint16).view(np.float16)[0]
                assert float(lo) == oracle.float_value(c, e, m) * 2.0 ** (bias - 15)
                assert float(hi) == oracle.float_value(c2, e, m) * 2.0 ** (bias - 15)
