"""Pins for the metadata-builder oracle (oracle/metadata.py).

The builder restates qsa_cache.py (_build_qsa_metadata_kernel and its torch
twin, _logical_positions, circular_qsa_slot_mapping,
compressed_qsa_slot_mapping).  Independent checks:
  * a hand-worked example: every output value derived by hand from the
    page's formulas (the arithmetic is in the comments);
  * closed forms of plain decode (one token per request at seq_len-1);
  * counting definitions: visible blocks = number of compression groups
    whose closing token 4g+3 is both at or before the row's position and
    inside the sequence; work items per request = number of groups closed
    inside the request's query chunk (at least one when it has queries);
  * invariants: positions are consecutive within a request and end at
    seq_len-1; a compressed slot points at exactly the page entry the
    selection reads for that group; circular slots are the query's last
    ``circular_buffer_size`` tokens and never collide.
"""
import numpy as np
import pytest

from oracle import metadata as M

# ---- hand-worked example -------------------------------------------------
# 5 requests; request 1 has no query tokens; tokens 12, 13 are padding.
#   query_start_loc = [0, 5, 5, 9, 11, 12], seq_lens = [20, 5, 8, 12, 28]
#   token -> request: t0..4 -> 0, t5..8 -> 2 (request 1 starts at 5 too but
#   is empty: the last request starting at or before t5 is 2), t9..10 -> 3,
#   t11 -> 4; padding -> 0.
#   position = seq_len - query_len + offset: request 0: 20-5+{0..4} = 15..19;
#   request 2: 8-4+{0..3} = 4..7; request 3: 12-2+{0,1} = 10, 11;
#   request 4: 28-1 = 27; padding -1.
QSL = [0, 5, 5, 9, 11, 12]
SL = [20, 5, 8, 12, 28]
BT = np.array([[5, 6, 4], [7, -1, -1], [3, -1, 9], [2, -1, 9], [1, 0, 8]], np.int32)
COMMON = [10, 11, 12, 13, -1, 15, 16, 17, 18, 19, 20, 21, 22, 23]
T2R = [0, 0, 0, 0, 0, 2, 2, 2, 2, 3, 3, 4, 0, 0]
LPOS = [15, 16, 17, 18, 19, 4, 5, 6, 7, 10, 11, 27, -1, -1]
# visible = max(0, min((pos+1)//4, L//4)): request 0 (L//4 = 5): 16//4 .. 20//4
# = 4,4,4,4,5; request 2 (L//4 = 2): 5//4..8//4 = 1,1,1,2; request 3 (3):
# 11//4, 12//4 = 2,3; request 4: min(28//4, 28//4) = 7.
VIS4 = [4, 4, 4, 4, 5, 1, 1, 1, 2, 2, 3, 7, 0, 0]
# compressed slots, compress_ratio 4, 2 keys per page: closing tokens are the
# positions 15, 19, 7, 11, 27 (t0, t4, t8, t10, t11).
#   t0: g = 3, column 1, page 6, common slot 10 >= 0 -> 6*2 + 1 = 13
#   t4: g = 4, column 2, page 4, but its common slot is -1 -> pad
#   t8: g = 1, column 0, page 3 -> 3*2 + 1 = 7
#   t10: g = 2, column 1, page -1 -> pad
#   t11: g = 6, column 3, past the 3-column table -> pad
SLOT_CMP = [13, -1, -1, -1, -1, -1, -1, -1, 7, -1, -1, -1, -1, -1]
# circular ring of 3 tokens in column 0's block; a token writes when
# t + 3 >= its request's query end; slot = block*3 + pos % 3:
#   request 0 (end 5, block 5): t2..t4, positions 17, 18, 19 -> 17, 15, 16
#   request 2 (end 9, block 3): t6..t8, positions 5, 6, 7   -> 11, 9, 10
#   request 3 (end 11, block 2): t9, t10, positions 10, 11  -> 7, 8
#   request 4 (end 12, block 1): t11, position 27           -> 3
SLOT_CIRC = [-1, -1, 17, 15, 16, -1, 11, 9, 10, 7, 8, 3, -1, -1]
# work items (compress_ratio 4): groups closed inside each query chunk
#   request 0: chunk [15, 19] closes groups 3 (15) and 4 (19) -> 2 items
#   request 1: no queries -> 0; request 2: [4, 7] closes group 1 -> 1
#   request 3: [10, 11] closes group 2 -> 1; request 4: [27] closes 6 -> 1
WORK7 = [(0, 0), (0, 1), (2, 0), (3, 0), (4, 0), (-1, -1), (-1, -1)]


def test_hand_worked_example_compressed():
    m = M.build_metadata(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=4,
                         common_slot_mapping=COMMON, max_num_work=7)
    assert m["token_to_req"].tolist() == T2R
    assert m["logical_positions"].tolist() == LPOS
    assert m["visible_blocks"].tolist() == VIS4
    assert m["slot_mapping"].tolist() == SLOT_CMP
    assert [tuple(x) for x in m["work_metadata"].tolist()] == WORK7
    assert m["work_total"] == 5


def test_hand_worked_example_circular_and_passthrough():
    m = M.build_metadata(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=4,
                         circular_buffer_size=3, common_slot_mapping=COMMON)
    assert m["slot_mapping"].tolist() == SLOT_CIRC
    m1 = M.build_metadata(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=1,
                          common_slot_mapping=COMMON)
    assert m1["slot_mapping"].tolist() == COMMON
    # compress_ratio 1: visible = min(pos+1, L) = pos+1 for every mapped token
    assert m1["visible_blocks"].tolist() == [p + 1 for p in LPOS[:12]] + [0, 0]


def test_truncated_work_list():
    m = M.build_metadata(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=4,
                         common_slot_mapping=COMMON, max_num_work=3)
    assert [tuple(x) for x in m["work_metadata"].tolist()] == WORK7[:3]


# ---- closed forms --------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_plain_decode_closed_form(seed):
    rng = np.random.default_rng(seed)
    R = 37
    L = rng.integers(1, 5000, size=R)
    cols = int(L.max() // 4 // 128 + 1)
    bt = rng.permutation(R * cols).astype(np.int32).reshape(R, cols)
    qsl = np.arange(R + 1)
    m = M.build_metadata(qsl, L, bt, R + 3, storage_block_size=128, compress_ratio=4,
                         common_slot_mapping=np.arange(R + 3), max_num_work=2 * R)
    assert m["token_to_req"].tolist() == list(range(R)) + [0, 0, 0]
    assert m["logical_positions"].tolist() == [int(x) - 1 for x in L] + [-1] * 3
    assert m["visible_blocks"].tolist() == [int(x) // 4 for x in L] + [0] * 3
    for i in range(R):
        s = int(m["slot_mapping"][i])
        if L[i] % 4 == 0:              # the new token closes group L/4 - 1
            g = int(L[i]) // 4 - 1
            assert s == int(bt[i, g // 128]) * 128 + g % 128
        else:
            assert s == -1
    # one work item per request: a group closes at L-1 or none does (then 1)
    assert [tuple(x) for x in m["work_metadata"][:R].tolist()] == [(i, 0) for i in range(R)]
    assert (m["work_metadata"][R:] == -1).all()


# ---- counting definitions and invariants on random batches ----------------
def _random_batch(rng, num_reqs, max_q, max_len, empty_frac=0.2):
    ql = rng.integers(1, max_q + 1, size=num_reqs)
    ql[rng.random(num_reqs) < empty_frac] = 0
    L = np.array([int(rng.integers(q, max_len + 1)) if q else int(rng.integers(0, max_len))
                  for q in ql])
    qsl = np.concatenate([[0], np.cumsum(ql)])
    return qsl, L, ql


@pytest.mark.parametrize("seed", range(6))
def test_counting_definitions(seed):
    rng = np.random.default_rng(100 + seed)
    num_reqs = int(rng.integers(1, 40))
    qsl, L, ql = _random_batch(rng, num_reqs, max_q=9, max_len=3000)
    sbs, cr = 16, 4
    cols = int(L.max() // cr // sbs + 1)
    bt = rng.permutation(num_reqs * cols + 7)[:num_reqs * cols].astype(np.int32)
    bt = bt.reshape(num_reqs, cols)
    bt[rng.random(bt.shape) < 0.1] = -1
    T = int(qsl[-1]) + int(rng.integers(0, 5))
    common = rng.integers(-1, 1000, size=T)
    maxw = int(rng.integers(0, 3 * num_reqs + 2))
    m = M.build_metadata(qsl, L, bt, T, storage_block_size=sbs, compress_ratio=cr,
                         common_slot_mapping=common, max_num_work=maxw)
    n_mapped = int(qsl[-1])
    for t in range(T):
        req = int(m["token_to_req"][t])
        lp = int(m["logical_positions"][t])
        if t >= n_mapped:
            assert (req, lp, int(m["visible_blocks"][t]), int(m["slot_mapping"][t])) == \
                (0, -1, 0, -1)
            continue
        assert qsl[req] <= t < qsl[req + 1]          # t lies in its request's query
        Lr = int(L[req])
        assert lp == Lr - int(ql[req]) + (t - int(qsl[req]))
        # visible blocks by counting closed groups
        vis = sum(1 for g in range(Lr) if 4 * g + 3 <= lp and 4 * g + 3 <= Lr - 1)
        assert int(m["visible_blocks"][t]) == vis
        # compressed slot: written only by a closing token, at the page entry
        # the selection reads for group g (page table column g // sbs)
        s = int(m["slot_mapping"][t])
        closes = lp >= 0 and lp % 4 == 3
        if s >= 0:
            assert closes and common[t] >= 0
            g = (lp - 3) // 4
            assert g // sbs < cols and bt[req, g // sbs] >= 0
            assert s // sbs == bt[req, g // sbs] and s % sbs == g % sbs
        elif closes and common[t] >= 0:
            g = (lp - 3) // 4
            assert g // sbs >= cols or bt[req, g // sbs] < 0
    # positions within a request: consecutive and ending at L-1
    for i in range(num_reqs):
        if ql[i]:
            seg = m["logical_positions"][qsl[i]:qsl[i + 1]].tolist()
            assert seg == list(range(int(L[i]) - int(ql[i]), int(L[i])))
    # work items by counting groups closed inside each query chunk
    expect = []
    for i in range(num_reqs):
        if not ql[i]:
            continue
        cs = int(L[i]) - int(ql[i])
        n = sum(1 for g in range(int(L[i])) if cs <= 4 * g + 3 <= int(L[i]) - 1)
        expect += [(i, j) for j in range(max(n, 1))]
    assert m["work_total"] == len(expect)
    got = [tuple(x) for x in m["work_metadata"].tolist()]
    assert got == (expect + [(-1, -1)] * maxw)[:maxw]


@pytest.mark.parametrize("cbs", [1, 4, 7])
def test_circular_ring_invariants(cbs):
    rng = np.random.default_rng(cbs)
    num_reqs = 23
    qsl, L, ql = _random_batch(rng, num_reqs, max_q=12, max_len=900)
    bt = rng.permutation(num_reqs).astype(np.int32).reshape(num_reqs, 1)
    bt[3, 0] = -1
    T = int(qsl[-1])
    m = M.build_metadata(qsl, L, bt, T, storage_block_size=64, compress_ratio=4,
                         circular_buffer_size=cbs)
    for i in range(num_reqs):
        seg = m["slot_mapping"][qsl[i]:qsl[i + 1]]
        n_write = 0 if bt[i, 0] < 0 else min(cbs, int(ql[i]))
        assert (seg[:len(seg) - n_write] == -1).all()
        w = seg[len(seg) - n_write:]
        assert (w >= 0).all()
        assert (w // cbs == bt[i, 0]).all()
        assert len(set(w.tolist())) == len(w)        # no two tokens share a ring slot
        lp = m["logical_positions"][qsl[i] + len(seg) - n_write:qsl[i + 1]]
        assert ((w % cbs) == (lp % cbs)).all()


def test_token_search_matches_linear_scan_with_many_empty_requests():
    rng = np.random.default_rng(9)
    ql = rng.integers(0, 3, size=300)
    ql[:5] = 0
    ql[-7:] = 0
    qsl = np.concatenate([[0], np.cumsum(ql)])
    L = ql + rng.integers(0, 100, size=300)
    m = M.build_metadata(qsl, L, np.zeros((300, 1), np.int32), int(qsl[-1]),
                         storage_block_size=8, compress_ratio=4)
    for t in range(int(qsl[-1])):
        owners = [i for i in range(300) if qsl[i] <= t < qsl[i + 1]]
        assert owners == [int(m["token_to_req"][t])]
