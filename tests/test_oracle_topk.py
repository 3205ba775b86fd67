"""Pins of the oracle's top-k page selection: hand-worked cases from
tests/golden, selection properties on random inputs with heavy ties, a
vectorised numpy formulation (lexsort), and head-group invariances."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    cases = []
    with open(os.path.join(GOLDEN, "topk_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals, sel = [x.strip() for x in line.split("|")]
            L, k, local = (int(x) for x in head.split())
            v = [(-np.inf if x == "-" else float(x)) for x in vals.split()]
            cases.append((L, k, local, v, [int(x) for x in sel.split()]))
    return cases


def _run(L, k, local, page_vals, rng, kv_groups=1):
    P = len(page_vals)
    sc = np.full((1, 64, P), -np.inf, dtype=np.float32)
    for j, v in enumerate(page_vals):
        if np.isfinite(v):
            # the page value sits on one random head; the others are lower
            h = rng.integers(0, 64)
            sc[0, :, j] = v - 1.0 - rng.random(64).astype(np.float32)
            sc[0, h, j] = v
    bt = (np.arange(P, dtype=np.int32) * 7 + 3).reshape(1, P)      # physical id of page j = 7j + 3
    sel, cnt = oracle.topk(decode=True, scores=sc, block_table=bt, block_table_stride=P, seq_lens=[L],
                           max_seq_len=P * 128, topk=k, local=local, kv_groups=kv_groups)
    return sel, cnt, bt


def test_golden_cases():
    rng = np.random.default_rng(0)
    cases = _golden()
    assert len(cases) == 9
    for L, k, local, v, want in cases:
        sel, cnt, bt = _run(L, k, local, v, rng)
        assert cnt[0, 0] == len(want), (L, k, local, v)
        assert list(sel[0, 0, :len(want)]) == [int(bt[0, j]) for j in want]
        assert (sel[0, 0, len(want):] == -1).all()


def _lexsort_select(vals, nl, k, local):
    """Vectorised restatement: forced tail, then np.lexsort on (index, -value)."""
    forced = min(local, nl)
    idx = np.arange(nl - forced)
    order = np.lexsort((idx, -vals[: nl - forced]))
    chosen = set(idx[order[: max(0, k - forced)]].tolist()) | set(range(nl - forced, nl))
    return sorted(chosen)


@pytest.mark.parametrize("kv_groups", [1, 2, 4])
def test_random_rows_with_ties(kv_groups):
    rng = np.random.default_rng(kv_groups)
    for _ in range(60):
        P = int(rng.integers(1, 40))
        L = int(rng.integers(0, P * 128 + 1))
        k = int(rng.integers(1, 12))
        local = int(rng.integers(0, k + 1))
        # values from a small set -> many ties
        sc = rng.integers(-3, 4, size=(1, 64, P)).astype(np.float32)
        nl = (L + 127) // 128
        sc[0, :, nl:] = -np.inf
        bt = rng.permutation(1000)[:P].astype(np.int32).reshape(1, P)
        sel, cnt = oracle.topk(decode=True, scores=sc, block_table=bt, block_table_stride=P, seq_lens=[L],
                               max_seq_len=P * 128, topk=k, local=local, kv_groups=kv_groups)
        hg = 64 // kv_groups
        for g in range(kv_groups):
            vals = sc[0, g * hg:(g + 1) * hg, :].max(axis=0).astype(np.float64)
            want = _lexsort_select(vals, nl, k, local)
            assert cnt[0, g] == len(want) == min(k, nl)
            assert list(sel[0, g, :len(want)]) == [int(bt[0, j]) for j in want]
            assert (sel[0, g, len(want):] == -1).all()
            # selection property: no unselected candidate beats a selected one
            forced = min(local, nl)
            cand = set(range(nl - forced))
            chosen = set(want) & cand
            for s in chosen:
                for u in cand - chosen:
                    assert vals[s] > vals[u] or (vals[s] == vals[u] and s < u)


def test_heads_matter_only_within_their_group():
    rng = np.random.default_rng(5)
    P, L = 12, 12 * 128
    sc = rng.normal(size=(1, 64, P)).astype(np.float32)
    bt = np.arange(P, dtype=np.int32).reshape(1, P)
    args = dict(decode=True, block_table=bt, block_table_stride=P, seq_lens=[L], max_seq_len=P * 128, topk=4,
                local=1, kv_groups=2)
    a, _ = oracle.topk(scores=sc, **args)
    # permuting heads inside each group changes nothing
    perm = np.concatenate([rng.permutation(32), 32 + rng.permutation(32)])
    b, _ = oracle.topk(scores=sc[:, perm, :], **args)
    np.testing.assert_array_equal(a, b)
    # a huge value on a group-1 head changes group 1 only
    sc2 = sc.copy()
    sc2[0, 40, 0] = 100.0
    c, _ = oracle.topk(scores=sc2, **args)
    np.testing.assert_array_equal(a[:, 0], c[:, 0])
    assert 0 in c[0, 1]


def test_prefill_rows_use_their_own_live_limit():
    """Row r of a request sees L = min(seq, prefix + pos + 1): later rows may
    have one more live page (and a different forced tail)."""
    P = 4
    sc = np.zeros((3, 64, P), dtype=np.float32)
    sc[:, :, 0] = 5.0
    bt = np.array([[20, 21, 22, 23]], dtype=np.int32)
    # prefix 254: row 0 sees 255 tokens (pages 0,1), row 1 256 (0,1), row 2 257 (0,1,2)
    sel, cnt = oracle.topk(decode=False, scores=sc, block_table=bt, block_table_stride=P, seq_lens=[257],
                           cu_seqlens_q=[0, 3], prefix_lens=[254], max_seq_len=512, topk=2, local=1)
    assert list(cnt[:, 0]) == [2, 2, 2]
    assert list(sel[0, 0]) == [20, 21] and list(sel[1, 0]) == [20, 21] and list(sel[2, 0]) == [20, 22]


@pytest.mark.parametrize("L", [1, 127, 128, 129, 1000, 1024, 4095])
def test_selected_tokens_special_cases(L):
    """The live-token count of the selected pages against what the selection
    fixes on its own: every live page taken gives the whole context L; only
    the forced tail page (topk 1) gives L's last page, L - 128 (ceil(L/128) -
    1); when every selected page is full (L a multiple of 128), 128 per page."""
    rng = np.random.default_rng(L)
    P = 32
    sc = rng.standard_normal((1, 64, P)).astype(np.float32)
    bt = np.arange(P, dtype=np.int32).reshape(1, P)
    nl = (L + 127) // 128
    kw = dict(decode=True, scores=sc, block_table=bt, block_table_stride=P, seq_lens=[L], max_seq_len=P * 128,
              want_tokens=True)
    _, cnt, tok = oracle.topk(topk=P, local=1, **kw)
    assert cnt[0, 0] == nl and tok[0, 0] == L
    _, cnt, tok = oracle.topk(topk=1, local=1, **kw)
    assert cnt[0, 0] == 1 and tok[0, 0] == L - 128 * (nl - 1)
    for k, local in ((3, 0), (5, 2)):
        _, cnt, tok = oracle.topk(topk=k, local=local, **kw)
        if L % 128 == 0:
            assert tok[0, 0] == 128 * cnt[0, 0]
        # a selection without the partial tail page is all full pages
        assert tok[0, 0] in (128 * cnt[0, 0], 128 * (cnt[0, 0] - 1) + L - 128 * (nl - 1))
