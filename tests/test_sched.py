"""Host-side schedulers (CPU only): coverage and makespan.

DISTFLASHATTN §4.5 (Fig. 4) quotes the ideal speedups of its schedules for
eight workers: 4.5x unbalanced and 7.2x balanced, i.e. 36 causal blocks
finished in 8 and in 5 steps (App. B, Figs. 5-6).  The fixture
tests/golden/balanced_schedule_fig4.json holds those printed numbers.
"""
import json
import os

import numpy as np
import pytest

from long_context_causal_gb300 import dfa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def blocks_of(P):
    return {qc * P + kc for qc in range(P) for kc in range(qc + 1)}


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16, 31, 32])
@pytest.mark.parametrize("sched", ["balanced", "unbalanced"])
def test_chunk_schedule_covers_every_causal_block_once(P, sched):
    st = dfa.dfa_chunk_schedule(P, sched)
    done = [int(b) for b in st.ravel() if b >= 0]
    assert len(done) == len(set(done)) == P * (P + 1) // 2
    assert set(done) == blocks_of(P)
    expect = P if sched == "unbalanced" else (P + 2) // 2
    assert st.shape[0] == expect


def test_chunk_schedule_matches_the_pages_fig4_speedups():
    with open(os.path.join(GOLDEN, "balanced_schedule_fig4.json")) as f:
        fx = json.load(f)
    P = fx["workers"]
    total = P * (P + 1) // 2
    unb = dfa.dfa_chunk_schedule(P, "unbalanced").shape[0]
    bal = dfa.dfa_chunk_schedule(P, "balanced").shape[0]
    assert total / unb == pytest.approx(fx["theoretical_speedup_unbalanced"])
    assert total / bal == pytest.approx(fx["theoretical_speedup_balanced"])


def test_balanced_helper_work_is_owned_by_a_mirror_worker():
    P = 8
    st = dfa.dfa_chunk_schedule(P, "balanced")
    for s in range(st.shape[0]):
        for w in range(P):
            b = st[s, w]
            if b < 0:
                continue
            qc = b // P
            assert qc == w or qc == P - 1 - w     # own chunk or the mirrored owner's


@pytest.mark.parametrize("rows,units,W", [(1, 4, 4), (32, 512, 148), (32, 1024, 152), (8, 512, 148),
                                          (3, 7, 5), (2, 1, 8), (1, 300, 148)])
@pytest.mark.parametrize("sched", ["balanced", "unbalanced"])
def test_worklist_covers_every_unit_once(rows, units, W, sched):
    off, items, mk = dfa.dfa_build_worklist(rows, units, W, sched)
    assert off[0] == 0 and off[-1] == rows * units and np.all(np.diff(off) >= 0)
    assert sorted(items.tolist()) == list(range(rows * units))
    cost = [sum(int(i) % units + 1 for i in items[off[w]:off[w + 1]]) for w in range(W)]
    assert mk == max(cost)
    # Rows are walked in order by every worker (L2 sharing of one head's K/V).
    for w in range(W):
        r = items[off[w]:off[w + 1]] // units
        assert np.all(np.diff(r) >= 0)


def test_balanced_worklist_beats_unbalanced_makespan():
    for rows, units, W in [(32, 512, 148), (32, 1024, 148), (8, 256, 148)]:
        _, _, mb = dfa.dfa_build_worklist(rows, units, W, "balanced")
        _, _, mu = dfa.dfa_build_worklist(rows, units, W, "unbalanced")
        ideal = rows * units * (units + 1) / 2 / W
        assert mb < mu
        assert mb <= ideal + units + 1          # within one mirror pair of perfect
        assert mu > 1.5 * ideal


def test_worklist_rejects_bad_arguments():
    with pytest.raises(dfa.DfaError):
        dfa.dfa_build_worklist(1, 4, 0)


# ---------------------------------------------------------------- split-kv helper items
def _hi(u, kv_tiles, causal):
    return min(2 * u + 2, kv_tiles) if causal else kv_tiles


@pytest.mark.parametrize("B,H,S,causal,n_sms", [(1, 1, 4096, True, 152), (1, 2, 8192, True, 152),
                                                (1, 1, 1000, True, 152), (1, 2, 2048, False, 152),
                                                (2, 3, 1536, True, 148), (1, 1, 32768, True, 152)])
def test_split_piece_tiles_gives_at_least_two_pieces_of_four_tiles(B, H, S, causal, n_sms):
    piece = dfa.dfa_split_piece_tiles(B, H, S, causal, n_sms)
    kv_tiles = -(-S // 128)
    assert piece >= 4
    assert -(-kv_tiles // piece) >= 2
    units = -(-S // 256)
    work = B * H * sum(_hi(u, kv_tiles, causal) for u in range(units))
    assert piece == max(4, -(-work // (2 * n_sms)))


@pytest.mark.parametrize("B,H,S,n_sms", [(1, 152, 4096, 152), (32, 32, 131072, 152), (1, 1, 256, 152),
                                         (1, 1, 384, 152), (0, 4, 1024, 152), (1, 4, 1024, 0)])
def test_split_is_not_used_when_every_sm_has_a_block_or_nothing_gains(B, H, S, n_sms):
    assert dfa.dfa_split_piece_tiles(B, H, S, True, n_sms) == 0


@pytest.mark.parametrize("rows,units,kv_tiles,causal,piece,W", [
    (1, 16, 32, True, 4, 152), (2, 32, 64, True, 7, 152), (1, 4, 8, True, 4, 10), (2, 8, 16, False, 4, 32),
    (6, 6, 12, True, 4, 36), (1, 128, 256, True, 55, 152), (3, 5, 9, True, 3, 7), (1, 1, 1, True, 4, 1)])
def test_split_worklist_covers_every_visible_tile_once(rows, units, kv_tiles, causal, piece, W):
    offsets, items, makespan = dfa.dfa_build_split_worklist(rows, units, kv_tiles, causal, piece, W)
    n_split = -(-kv_tiles // piece)
    assert offsets[0] == 0 and np.all(np.diff(offsets) >= 0) and offsets[-1] == len(items)
    assert len(set(items.tolist())) == len(items)
    seen = {}
    cost = []
    for w in range(W):
        c = 0
        for it in items[offsets[w]:offsets[w + 1]]:
            s, ru = int(it) % n_split, int(it) // n_split
            row, u = ru // units, ru % units
            assert 0 <= row < rows
            hi = _hi(u, kv_tiles, causal)
            lo, top = s * piece, min((s + 1) * piece, hi)
            assert lo < top, "empty pieces are not listed"
            for j in range(lo, top):
                key = (row, u, j)
                assert key not in seen
                seen[key] = w
            c += 2 * (top - lo)
        cost.append(c)
    expect = {(r, u, j) for r in range(rows) for u in range(units) for j in range(_hi(u, kv_tiles, causal))}
    assert set(seen) == expect
    assert makespan == max(cost)
    # Longest-first greedy: no worker ends more than one piece above the average.
    assert makespan <= sum(cost) / W + 2 * piece


def test_split_worklist_rejects_bad_arguments():
    for args in [(1, 4, 8, True, 0, 4), (1, 4, 8, True, 4, 0), (-1, 4, 8, True, 4, 4)]:
        with pytest.raises(dfa.DfaError):
            dfa.dfa_build_split_worklist(*args)


# ---------------------------------------------------------------- variable-length batches
@pytest.mark.parametrize("units,heads,causal,W", [([3, 0, 2], 2, True, 4), ([16, 1, 7, 8, 0, 33], 4, True, 152),
                                                  ([5, 5, 5], 2, False, 6), ([1], 1, True, 1),
                                                  ([64, 2, 2, 2, 2, 2, 2, 2], 8, True, 148)])
def test_varlen_worklist_covers_every_unit_once_and_keeps_mirror_pairs(units, heads, causal, W):
    umax = max(units)
    offsets, items, makespan = dfa.dfa_build_varlen_worklist(units, heads, umax, causal, W)
    assert offsets[0] == 0 and np.all(np.diff(offsets) >= 0) and offsets[-1] == len(items)
    expect = {(s * heads + h) * umax + u for s, n in enumerate(units) for h in range(heads) for u in range(n)}
    assert sorted(items.tolist()) == sorted(expect)
    cost = []
    for w in range(W):
        mine = items[offsets[w]:offsets[w + 1]].tolist()
        c = 0
        for it in mine:
            row, u = divmod(it, umax)
            n = units[row // heads]
            c += (u + 1) if causal else n
            if causal and u != n - 1 - u:
                assert (row * umax + (n - 1 - u)) in mine, "a unit travels with its mirror"
        cost.append(c)
    assert makespan == max(cost)
    biggest = max((n + 1) if causal else n for n in units if n) if any(units) else 0
    assert makespan <= sum(cost) / W + biggest


def test_varlen_workspace_and_worklist_reject_bad_offsets():
    assert dfa.dfa_attn_varlen_workspace_size([0, 100, 50], 4, 2, 128, True) == 0
    assert dfa.dfa_attn_varlen_workspace_size([1, 100], 4, 2, 128, False) == 0
    assert dfa.dfa_attn_varlen_workspace_size([0, 100], 4, 3, 128, False) == 0
    assert dfa.dfa_attn_varlen_workspace_size([0], 4, 2, 128, True) > 0
    with pytest.raises(dfa.DfaError):
        dfa.dfa_build_varlen_worklist([3, 5], 2, 4, True, 4)   # a sequence above n_units_max


# ---------------------------------------------------------------- backward split-kv
@pytest.mark.parametrize("B,Hkv,S,causal,n_sms", [(1, 1, 4096, True, 152), (1, 1, 8192, True, 152),
                                                  (1, 1, 16384, True, 152), (1, 1, 4096, False, 152),
                                                  (2, 1, 8192, True, 148)])
def test_split_bwd_piece_tiles(B, Hkv, S, causal, n_sms):
    piece = dfa.dfa_split_bwd_piece_tiles(B, Hkv, S, causal, n_sms)
    n = -(-S // 128)
    work = B * Hkv * (n * (n + 1) // 2 if causal else n * n)
    assert piece == max(16, -(-work // (2 * n_sms)))
    assert -(-n // piece) >= 2


@pytest.mark.parametrize("B,Hkv,S,n_sms", [(1, 32, 131072, 152), (1, 1, 1024, 152), (1, 8, 65536, 152), (0, 1, 4096, 152)])
def test_split_bwd_not_used_on_large_or_short_problems(B, Hkv, S, n_sms):
    assert dfa.dfa_split_bwd_piece_tiles(B, Hkv, S, True, n_sms) == 0


def test_split_bwd_needs_a_quarter_of_the_sms_idle():
    # 128 key tiles per row: 64 mirror pairs per row
    assert dfa.dfa_split_bwd_piece_tiles(1, 1, 16384, True, 152) > 0       # 64 pairs
    assert dfa.dfa_split_bwd_piece_tiles(1, 2, 16384, True, 152) == 0      # 128 pairs > 114
    assert dfa.dfa_split_bwd_piece_tiles(1, 1, 24576, True, 152) > 0       # 96 pairs


@pytest.mark.parametrize("rows,n,causal,piece,W", [(1, 32, True, 16, 152), (1, 64, True, 16, 152),
                                                   (1, 128, True, 28, 152), (2, 32, False, 16, 64), (3, 9, True, 4, 5)])
def test_bwd_split_worklist_covers_every_visible_tile_pair_once(rows, n, causal, piece, W):
    offsets, items, makespan = dfa.dfa_build_bwd_split_worklist(rows, n, causal, piece, W)
    n_split = -(-n // piece)
    assert offsets[0] == 0 and np.all(np.diff(offsets) >= 0) and offsets[-1] == len(items)
    seen, cost = set(), []
    for w in range(W):
        c = 0
        for it in items[offsets[w]:offsets[w + 1]].tolist():
            s, ru = it % n_split, it // n_split
            row, u = ru // n, ru % n
            t = n - 1 - u
            lo_i = t if causal else 0
            lo, hi = lo_i + s * piece, min(n, lo_i + (s + 1) * piece)
            assert lo < hi, "empty pieces are not listed"
            for i in range(lo, hi):
                assert (row, t, i) not in seen
                seen.add((row, t, i))
            c += hi - lo
        cost.append(c)
    assert seen == {(r, t, i) for r in range(rows) for t in range(n) for i in range(t if causal else 0, n)}
    assert makespan == max(cost)
    assert makespan <= sum(cost) / W + piece
