"""Host scheduler: the per-SM instruction queues cover every output exactly
once, dependency counts match the producers, queues respect one topological
order, and a simulator that executes the queues under random interleavings
with the kernel's counter semantics always completes (no deadlock)."""
import random
from collections import defaultdict

import numpy as np
import pytest

from decode_megakernel_llama_gb300 import _lib
from decode_megakernel_llama_gb300.build import build
from decode_megakernel_llama_gb300.configs import LLAMA_1B, LLAMA_3B, TINY, ModelShape

OP_QKV, OP_ATTN, OP_OPROJ, OP_GATEUP, OP_DOWN, OP_LMHEAD = 1, 2, 3, 4, 5, 6
F_OP, F_LAYER, F_A0, F_A1, F_MAT, F_WAIT, F_TGT, F_SIG, F_SIGN, F_STAGE, F_SLOT = range(11)

ODD = ModelShape("odd", 3, 768, 12, 4, 64, 3072, 1000, 1e-5, 1e4)

CASES = [(TINY, 152, 40), (TINY, 7, 40), (LLAMA_1B, 152, 256), (LLAMA_1B, 148, 8256),
         (LLAMA_3B, 152, 384), (ODD, 13, 300), (ODD, 1, 64)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def plan(shape, n_sm, max_seq):
    instr, qlen, nctr = _lib.plan_inspect(shape, n_sm, max_seq)
    assert qlen.sum() == len(instr)
    queues, k = [], 0
    for n in qlen:
        queues.append(instr[k:k + n])
        k += n
    return instr, queues, nctr


def cover(intervals, total):
    iv = sorted(intervals)
    pos = 0
    for a, n in iv:
        assert a == pos and n > 0, (a, pos, n)
        pos += n
    assert pos == total


@pytest.mark.parametrize("shape,n_sm,max_seq", CASES)
def test_every_output_row_exactly_once(shape, n_sm, max_seq):
    instr, _, _ = plan(shape, n_sm, max_seq)
    hd = shape.head_dim
    stacked = (shape.n_heads + 2 * shape.n_kv_heads) * hd  # rows of [Wq; Wk; Wv]
    by = defaultdict(list)
    for r in instr:
        op, l = int(r[F_OP]), int(r[F_LAYER])
        if op == OP_ATTN:
            by[(op, l, int(r[F_A0]), int(r[F_SLOT]))].append((int(r[F_A1]), 1))
        else:
            by[(op, l)].append((int(r[F_A0]), int(r[F_A1])))
    S = len(by[(OP_ATTN, 0, 0, 0)])
    assert S >= 1
    # the query heads of a kv head may be split over parts (slot 0 .. AP-1)
    AP = len({int(r[F_SLOT]) for r in instr if r[F_OP] == OP_ATTN})
    assert shape.n_heads // shape.n_kv_heads % AP == 0
    for l in range(shape.n_layers):
        cover(by[(OP_QKV, l)], stacked)
        for h in range(shape.n_kv_heads):
            for a in range(AP):
                cover(by[(OP_ATTN, l, h, a)], S)
        cover(by[(OP_OPROJ, l)], shape.d_model)
        cover(by[(OP_GATEUP, l)], shape.ffn_dim)
        cover(by[(OP_DOWN, l)], shape.d_model)
    cover(by[(OP_LMHEAD, 0)], shape.vocab)
    slots = sorted(int(r[F_SLOT]) for r in instr if r[F_OP] == OP_LMHEAD)
    assert slots == list(range(len(slots)))
    assert max(int(r[F_A1]) for r in instr if r[F_OP] != OP_ATTN) <= 2048


def test_query_heads_split_where_attention_is_on_the_critical_path():
    # one sequence, even group size, attention on few SMs: two instructions per
    # kv head; odd groups (3B-class) and long contexts (every SM busy) keep one
    parts = lambda *a: len({int(r[F_SLOT]) for r in plan(*a)[0] if r[F_OP] == OP_ATTN})
    assert parts(LLAMA_1B, 152, 256) == 2
    assert parts(LLAMA_3B, 152, 384) == 1
    assert parts(LLAMA_1B, 148, 8256) == 1
    instr, _, _ = _lib.plan_inspect(LLAMA_1B, 152, 1024, max_batch=8)
    assert {int(r[F_SLOT]) for r in instr if r[F_OP] == OP_ATTN} == {0}


def signal_counts(instr, shape, S):
    """How many times each counter is bumped in one step (kernel semantics)."""
    sig = defaultdict(int)
    for r in instr:
        for c in range(int(r[F_SIG]), int(r[F_SIG]) + int(r[F_SIGN])):
            sig[c] += 1
    return sig


@pytest.mark.parametrize("shape,n_sm,max_seq", CASES)
def test_wait_targets_equal_producer_counts_and_stages_ordered(shape, n_sm, max_seq):
    instr, queues, nctr = plan(shape, n_sm, max_seq)
    sig = signal_counts(instr, shape, None)
    producers_stage = defaultdict(set)
    for r in instr:
        for c in range(int(r[F_SIG]), int(r[F_SIG]) + int(r[F_SIGN])):
            producers_stage[c].add(int(r[F_STAGE]))
    L, Hkv = shape.n_layers, shape.n_kv_heads
    attn_done0 = 2 * L * Hkv  # counter layout: qkv_grp, merge, attn_done, ...
    for r in instr:
        c, tgt = int(r[F_WAIT]), int(r[F_TGT])
        if c < 0:
            assert r[F_OP] == OP_QKV and r[F_LAYER] == 0
            continue
        assert 0 <= c < nctr
        if attn_done0 <= c < attn_done0 + L:   # bumped by the last split of each kv head
            assert r[F_OP] == OP_OPROJ and tgt == Hkv
            continue
        assert tgt == sig[c] and tgt > 0, (r, sig[c])
        assert max(producers_stage[c]) < int(r[F_STAGE])
    for q in queues:
        st = [int(r[F_STAGE]) for r in q]
        assert st == sorted(st)


def simulate(instr, queues, nctr, shape, seed):
    """Execute the queues in a random interleaving; return True if all finish."""
    rng = random.Random(seed)
    ctr = [0] * nctr
    L, Hkv = shape.n_layers, shape.n_kv_heads
    S = sum(1 for r in instr if r[F_OP] == OP_ATTN and r[F_LAYER] == 0 and r[F_A0] == 0)
    merge0, attn_done0 = L * Hkv, 2 * L * Hkv
    ptr = [0] * len(queues)
    remaining = sum(len(q) for q in queues)
    while remaining:
        ready = [s for s, q in enumerate(queues) if ptr[s] < len(q)
                 and (q[ptr[s]][F_WAIT] < 0 or ctr[int(q[ptr[s]][F_WAIT])] >= int(q[ptr[s]][F_TGT]))]
        if not ready:
            return False
        s = rng.choice(ready)
        r = queues[s][ptr[s]]
        ptr[s] += 1
        remaining -= 1
        for c in range(int(r[F_SIG]), int(r[F_SIG]) + int(r[F_SIGN])):
            ctr[c] += 1
        if r[F_OP] == OP_ATTN:
            m = merge0 + int(r[F_LAYER]) * Hkv + int(r[F_A0])
            ctr[m] += 1
            if ctr[m] == S:
                ctr[attn_done0 + int(r[F_LAYER])] += 1
    return True


@pytest.mark.parametrize("shape,n_sm,max_seq", CASES)
def test_random_interleavings_never_deadlock(shape, n_sm, max_seq):
    instr, queues, nctr = plan(shape, n_sm, max_seq)
    for seed in range(3):
        assert simulate(instr, queues, nctr, shape, seed)


def test_simulator_catches_a_bad_order():
    # Planting a stage inversion in one queue (an O-projection ahead of its
    # attention) must deadlock the simulator when that SM is the only one.
    instr, queues, nctr = plan(TINY, 1, 40)
    q = list(queues[0])
    i_o = next(i for i, r in enumerate(q) if r[F_OP] == OP_OPROJ)
    i_a = next(i for i, r in enumerate(q) if r[F_OP] == OP_ATTN)
    q[i_a], q[i_o] = q[i_o], q[i_a]
    assert not simulate(instr, [np.array(q)], nctr, TINY, 0)


@pytest.mark.parametrize("shape,n_sm,max_seq", [(LLAMA_1B, 152, 256), (LLAMA_3B, 152, 384)])
def test_bytes_per_sm_are_balanced(shape, n_sm, max_seq):
    instr, queues, _ = plan(shape, n_sm, max_seq)
    per_sm = [sum(int(r[11]) + (int(r[12]) << 32) for r in q) for q in queues]
    total = sum(per_sm)
    assert total == shape.step_weight_bytes() - 2 * shape.d_model * (1 + 2 * shape.n_layers + 1) + 0 \
        or total > 0
    # attention SMs skip the QKV rows of their layer; the other ops even out
    # the bytes only up to one row each, so allow a few percent
    assert max(per_sm) / (total / n_sm) < 1.03


# ---- bulk-copy bounds (the producer's tile arithmetic, checked on the CPU) ----

PAGE, NPAGES, WARPS, REDCAP, DREDCAP, RESID, STAGED, STAGED_LONG = 32768, 6, 8, 2048, 256, 256, 4096, 8192


def geo(K):
    sw = 1
    while K // sw > 1024 or (K // sw) % 256:
        sw *= 2
    rw = WARPS // sw
    m = PAGE // (rw * K * 2)
    return dict(K=K, sw=sw, rw=rw, m=m, rt=rw * m, nx=K // sw // 32)


def attn_tiles(pos, S, ppt, split):
    need = max(1, (pos + ppt - 1) // ppt)
    seff = min(need, S)
    if split >= seff:
        return []
    chunk = (pos + seff - 1) // seff
    t0 = min(split * chunk, pos)
    t1 = min(t0 + chunk, pos)
    out, ts = [], t0
    while ts < t1:
        out.append((ts, min(ppt, t1 - ts)))
        ts += ppt
    return out


@pytest.mark.parametrize("shape,n_sm,max_seq", CASES)
def test_tile_copies_stay_in_bounds(shape, n_sm, max_seq):
    instr, _, _ = plan(shape, n_sm, max_seq)
    d, F, hd = shape.d_model, shape.ffn_dim, shape.head_dim
    qd, kvd = shape.n_heads * hd, shape.n_kv_heads * hd
    G = {OP_QKV: geo(d), OP_OPROJ: geo(qd), OP_GATEUP: geo(d), OP_DOWN: geo(F), OP_LMHEAD: geo(d)}
    mat_rows = {OP_QKV: qd + 2 * kvd, OP_OPROJ: d, OP_GATEUP: F, OP_DOWN: d, OP_LMHEAD: shape.vocab}
    assert d <= STAGED and qd <= STAGED and F <= STAGED_LONG
    ppt = (PAGE // 2) // (hd * 2)
    S = sum(1 for r in instr if r[F_OP] == OP_ATTN and r[F_LAYER] == 0 and r[F_A0] == 0 and r[F_SLOT] == 0)
    for r in instr:
        op = int(r[F_OP])
        if op == OP_ATTN:
            for pos in sorted({0, 1, ppt - 1, ppt, ppt + 1, max_seq // 2, max_seq - 1}):
                if not 0 <= pos < max_seq:
                    continue
                covered = []
                for ts, n in attn_tiles(pos, S, ppt, int(r[F_A1])):
                    assert 0 < n <= ppt and ts + n <= pos < max_seq
                    assert (n * hd * 2) % 16 == 0 and n * hd * 2 <= PAGE // 2
                    covered.append((ts, n))
            continue
        g = G[op]
        per = g["rt"] // 2 if op == OP_GATEUP else g["rt"]
        assert per >= 1 and g["m"] >= 1 and g["nx"] in (8, 16, 24, 32)
        n, a0 = int(r[F_A1]), int(r[F_A0])
        nrows = mat_rows[op]
        nt = -(-n // per)
        for j in range(nt):
            rows = min(per, n - j * per)
            row0 = a0 + j * per
            nbytes = rows * g["K"] * 2
            assert rows > 0 and nbytes % 16 == 0
            assert (row0 + rows) <= nrows
            dst1 = per * g["K"] * 2 if op == OP_GATEUP else 0
            assert dst1 + nbytes <= PAGE
            if op == OP_QKV:
                # a stacked-QKV tile crossing a matrix boundary is two copies
                for b in (qd, qd + kvd):
                    if row0 < b < row0 + rows:
                        assert ((b - row0) * g["K"] * 2) % 16 == 0
                        assert ((row0 + rows - b) * g["K"] * 2) % 16 == 0
                assert sum(row0 < b < row0 + rows for b in (qd, qd + kvd)) <= 1
        # per-row partials fit their reduction buffer, residual rows theirs
        outs = 2 * n if op == OP_GATEUP else n
        assert outs * g["sw"] <= (DREDCAP if op == OP_DOWN else REDCAP)
        if op in (OP_OPROJ, OP_DOWN):
            assert n <= RESID


def test_attention_splits_cover_every_cached_position():
    for pos in range(0, 700, 7):
        for S in (1, 2, 3, 5, 19):
            got = []
            last_active = None
            for s in range(S):
                t = attn_tiles(pos, S, 128, s)
                got += [p for ts, n in t for p in range(ts, ts + n)]
            assert got == list(range(pos)), (pos, S)


# ---- the fused batched step's plan (max_batch > 1) ----

BATCH_CASES = [(TINY, 152, 40, 3), (TINY, 16, 24, 2), (TINY, 5, 24, 2), (LLAMA_1B, 152, 1024, 8), (LLAMA_1B, 148, 600, 4)]


def simulate_batch(instr, queues, nctr, shape, nb, seed):
    """As simulate(), with one merge per (sequence, layer, kv head)."""
    rng = random.Random(seed)
    ctr = [0] * nctr
    L, Hkv = shape.n_layers, shape.n_kv_heads
    S = sum(1 for r in instr if r[F_OP] == OP_ATTN and r[F_LAYER] == 0 and r[F_A0] == 0 and r[F_MAT] == 0)
    attn_done0 = 2 * L * Hkv
    merged = defaultdict(int)
    ptr = [0] * len(queues)
    remaining = sum(len(q) for q in queues)
    while remaining:
        ready = [s for s, q in enumerate(queues) if ptr[s] < len(q)
                 and (q[ptr[s]][F_WAIT] < 0 or ctr[int(q[ptr[s]][F_WAIT])] >= int(q[ptr[s]][F_TGT]))]
        if not ready:
            return False
        s = rng.choice(ready)
        r = queues[s][ptr[s]]
        ptr[s] += 1
        remaining -= 1
        for c in range(int(r[F_SIG]), int(r[F_SIG]) + int(r[F_SIGN])):
            ctr[c] += 1
        if r[F_OP] == OP_ATTN:
            key = (int(r[F_MAT]), int(r[F_LAYER]), int(r[F_A0]))
            merged[key] += 1
            if merged[key] == S:
                ctr[attn_done0 + int(r[F_LAYER])] += 1
    return True


@pytest.mark.parametrize("shape,n_sm,max_seq,nb", BATCH_CASES)
def test_batched_plan_covers_every_row_and_sequence(shape, n_sm, max_seq, nb):
    instr, qlen, nctr = _lib.plan_inspect(shape, n_sm, max_seq, max_batch=nb)
    hd, d, F = shape.head_dim, shape.d_model, shape.ffn_dim
    stacked = (shape.n_heads + 2 * shape.n_kv_heads) * hd
    by = defaultdict(list)
    for r in instr:
        op, l = int(r[F_OP]), int(r[F_LAYER])
        if op == OP_ATTN:
            by[(op, l, int(r[F_A0]), int(r[F_MAT]))].append((int(r[F_A1]), 1))
        else:
            assert int(r[F_MAT]) == 0
            by[(op, l)].append((int(r[F_A0]), int(r[F_A1])))
    S = len(by[(OP_ATTN, 0, 0, 0)])
    assert S >= 1
    assert not any(k[0] == OP_ATTN and k[3] >= nb for k in by)
    for l in range(shape.n_layers):
        cover(by[(OP_QKV, l)], stacked)
        for b in range(nb):
            for h in range(shape.n_kv_heads):
                cover(by[(OP_ATTN, l, h, b)], S)
        cover(by[(OP_OPROJ, l)], d)
        cover(by[(OP_GATEUP, l)], F)
        cover(by[(OP_DOWN, l)], d)
    # the batched LM head is a tensor-core contraction after the launch
    assert not any(int(r[F_OP]) == OP_LMHEAD for r in instr)
    # shared-memory capacities of the batched GEMV: accumulators for all 8
    # sequence lanes of every output row (two per row for gate/up), and the
    # residual rows of every sequence for O-proj and down
    for r in instr:
        op, n = int(r[F_OP]), int(r[F_A1])
        if op in (OP_QKV, OP_OPROJ, OP_DOWN):
            assert n * 8 <= REDCAP
        if op == OP_GATEUP:
            assert 2 * n * 8 <= REDCAP
        if op in (OP_OPROJ, OP_DOWN):
            assert n * nb <= RESID
    queues, k = [], 0
    for q in qlen:
        queues.append(instr[k:k + q])
        k += q
    for seed in range(2):
        assert simulate_batch(instr, queues, nctr, shape, nb, seed)


def batch_geo(K):
    KC = min(K, 1024)
    sw = KC // 128
    return dict(K=K, KC=KC, sw=sw, rt=(WARPS // sw) * 16)


@pytest.mark.parametrize("shape,n_sm,max_seq,nb", BATCH_CASES)
def test_batched_tile_copies_stay_in_bounds(shape, n_sm, max_seq, nb):
    # tile = rt rows x a K-chunk of KC columns; a K-chunked tile is copied
    # row by row (KC*2 bytes each, 16-byte aligned); every warp's 16 rows and
    # 128-wide slice lie inside the tile
    instr, _, _ = _lib.plan_inspect(shape, n_sm, max_seq, max_batch=nb)
    d, F, hd = shape.d_model, shape.ffn_dim, shape.head_dim
    qd, kvd = shape.n_heads * hd, shape.n_kv_heads * hd
    G = {OP_QKV: batch_geo(d), OP_OPROJ: batch_geo(qd), OP_GATEUP: batch_geo(d), OP_DOWN: batch_geo(F)}
    mat_rows = {OP_QKV: qd + 2 * kvd, OP_OPROJ: d, OP_GATEUP: F, OP_DOWN: d}
    for r in instr:
        op = int(r[F_OP])
        if op == OP_ATTN:
            continue
        g = G[op]
        assert g["K"] % g["KC"] == 0 and g["rt"] * g["KC"] * 2 <= PAGE and (g["KC"] * 2) % 16 == 0
        per = g["rt"] // 2 if op == OP_GATEUP else g["rt"]
        n, a0 = int(r[F_A1]), int(r[F_A0])
        for j in range(-(-n // per)):
            rows = min(per, n - j * per)
            assert rows > 0 and a0 + j * per + rows <= mat_rows[op]
        # warp (rg, ks): rows rg*16 .. +16 (gate/up: rg*8 .. +8 of each half), columns ks*128 .. +128
        for w in range(WARPS):
            rg, ks = w // g["sw"], w % g["sw"]
            assert (ks + 1) * 128 <= g["KC"]
            if op == OP_GATEUP:
                assert per + rg * 8 + 8 <= g["rt"]
            else:
                assert rg * 16 + 16 <= g["rt"]


def test_batched_plan_falls_back_where_unsupported():
    # head_dim 128 has no batched kernel instance: the single-sequence plan
    # (no attention for sequences > 0)
    for shape, n_sm in ((LLAMA_3B, 152),):
        instr, _, _ = _lib.plan_inspect(shape, n_sm, 64, max_batch=2)
        assert not any(int(r[F_MAT]) > 0 for r in instr if r[F_OP] == OP_ATTN)
        single, _, _ = _lib.plan_inspect(shape, n_sm, 64)
        assert np.array_equal(instr, single)


def test_lm_head_blocks_and_the_filtered_draw_path():
    # The last LM-head block sorts up to 16384 candidate keys (64 per block):
    # Llama-1B's 152 blocks draw in the epilogue; the 3B-class d_model 3072
    # splits each SM's 844 rows in two (512 rows per block at most), 304
    # blocks, so its filtered draw runs after the launch.
    for shape, inside in ((LLAMA_1B, True), (LLAMA_3B, False)):
        instr, _, _ = _lib.plan_inspect(shape, 152, 64)
        n_lm = int((instr[:, F_OP] == OP_LMHEAD).sum())
        assert (n_lm * 64 <= 16384) == inside, (shape.name, n_lm)
