"""zf_kv, the host-side page manager (CPU only: bookkeeping, no GPU calls).

ZipFusion §III.D: pages stay uncompressed while they fill, a full page is compressed afterwards
under its page id, new pages are counted in uncompressed storage until compression releases it,
and storage released in one layer can be reassigned to another.  The checks below restate those
rules as invariants of the manager's state and run a random workload against a plain Python model
of the same rules, with one layer and with several layers sharing one raw-slot pool."""
import random

import pytest

from tests import helpers as H


@pytest.fixture(scope="module")
def zf():
    return H.zf_module()


P = 16


def test_admit_lists_every_page_for_an_uncompressed_first_write(zf):
    kv = zf.KvManager(num_pages=10, num_raw_slots=10, page_size=P, max_requests=4, max_pages_per_req=8)
    ids, nv, rs = kv.admit(0, 37)
    assert ids == [0, 1, 2] and nv == [16, 16, 5] and rs == [[0, 1, 2]]
    st = kv.stats()
    assert (st["free_pages"], st["free_raw_slots"], st["pending_pages"], st["partial_pages"]) == (7, 7, 2, 1)
    assert st["tokens"] == 37 and st["new_page_capacity"] == 7
    table, lens = kv.export()
    assert table[0, :4].tolist() == [0, 1, 2, -1] and lens.tolist() == [37, 0, 0, 0]
    # the two full pages are reported compressed: their raw slots come back
    pend, slots = kv.pending()
    assert pend == [0, 1] and slots == [[0, 1]]
    kv.reclaim(pend, [[False, False]])
    st = kv.stats()
    assert (st["free_raw_slots"], st["pending_pages"], st["compressed_pages"]) == (9, 0, 2)


def test_append_fills_the_tail_then_opens_a_new_page(zf):
    kv = zf.KvManager(num_pages=6, num_raw_slots=3, page_size=P, max_requests=2, max_pages_per_req=6)
    kv.admit(0, 14)                                   # one partial page, raw slot 0
    for expect_fill in (15, 16):
        ids, nv, rs = kv.append([0])
        assert ids == [0] and nv == [expect_fill] and rs == [[0]]
    assert kv.stats()["pending_pages"] == 1 and kv.stats()["partial_pages"] == 0
    ids, nv, rs = kv.append([0])                       # token 17 opens page 1 with a new raw slot
    assert ids == [1] and nv == [1] and rs == [[1]]
    kv.reclaim([0], [[True]])                          # page 0 stayed raw: keeps slot 0
    st = kv.stats()
    assert st["raw_full_pages"] == 1 and st["raw_full_slots"] == 1 and st["free_raw_slots"] == 1
    kv.release(0)
    st = kv.stats()
    assert (st["free_pages"], st["free_raw_slots"], st["active_requests"], st["tokens"]) == (6, 3, 0, 0)


def test_capacity_refusals_change_nothing(zf):
    kv = zf.KvManager(num_pages=5, num_raw_slots=3, page_size=P, max_requests=3, max_pages_per_req=4)
    kv.admit(0, 32)                                    # 2 ids, 2 raw slots (pending)
    before = kv.stats()
    with pytest.raises(zf.ZfError, match="page ids or raw slots"):
        kv.admit(1, 40)                                # 3 pages but 1 raw slot free
    assert kv.stats() == before and kv.export()[1][1] == 0
    kv.admit(1, 16)                                    # exactly one page: fits
    with pytest.raises(zf.ZfError, match="page ids or raw slots"):
        kv.append([0, 1])                              # both open a page: 2 ids free, no raw slot
    assert kv.stats()["tokens"] == 48
    ids, _ = kv.pending()
    kv.reclaim(ids, [[False] * len(ids)])              # compression releases uncompressed storage
    ids, nv, rs = kv.append([0, 1])
    assert nv == [1, 1] and len(set(rs[0])) == 2


def test_invalid_calls_are_refused(zf):
    kv = zf.KvManager(num_pages=4, num_raw_slots=4, page_size=P, max_requests=2, max_pages_per_req=2)
    kv.admit(0, 5)
    with pytest.raises(zf.ZfError):
        kv.admit(0, 5)                                 # slot already active
    with pytest.raises(zf.ZfError):
        kv.admit(1, 33)                                # more pages than a request may hold
    with pytest.raises(zf.ZfError):
        kv.append([1])                                 # inactive request
    with pytest.raises(zf.ZfError):
        kv.append([0, 0])                              # the same request twice
    with pytest.raises(zf.ZfError):
        kv.reclaim([0], [[False]])                     # page 0 is partial, not pending
    with pytest.raises(zf.ZfError):
        kv.release(1)


def test_raw_slots_freed_in_one_layer_serve_another(zf):
    """Three layers share a pool of 9 raw slots: a new page takes one slot per layer; after the
    encodes, a layer that compressed the page returns its slot and a layer that left it raw keeps
    only its own; the freed slots open new pages for every layer."""
    kv = zf.KvManager(num_pages=10, num_raw_slots=9, page_size=P, max_requests=3, max_pages_per_req=6, num_layers=3)
    ids, nv, rs = kv.admit(0, 40)                      # 3 pages x 3 layers: the whole pool
    assert ids == [0, 1, 2] and nv == [16, 16, 8]
    assert sorted(s for row in rs for s in row) == list(range(9)) and [len(row) for row in rs] == [3, 3, 3]
    st = kv.stats()
    assert (st["free_raw_slots"], st["new_page_capacity"], st["pending_pages"]) == (0, 0, 2)
    with pytest.raises(zf.ZfError, match="page ids or raw slots"):
        kv.admit(1, 1)
    pend, slots = kv.pending()
    assert pend == [0, 1] and slots == [[rs[l][0], rs[l][1]] for l in range(3)]
    # page 0 stays raw in layer 2 only; page 1 compresses everywhere
    kv.reclaim(pend, [[False, False], [False, False], [True, False]])
    st = kv.stats()
    assert (st["free_raw_slots"], st["raw_full_pages"], st["raw_full_slots"], st["compressed_pages"]) == (5, 1, 1, 1)
    assert st["new_page_capacity"] == 1               # 5 slots: one page in all three layers
    ids1, _, rs1 = kv.admit(1, 16)
    freed = {rs[l][0] for l in range(2)} | {rs[l][1] for l in range(3)}
    assert {row[0] for row in rs1} <= freed and len({row[0] for row in rs1}) == 3
    kv.release(0)                                      # the kept slot and the tail's slots come back
    st = kv.stats()
    assert (st["free_raw_slots"], st["raw_full_pages"], st["raw_full_slots"]) == (6, 0, 0)


def test_per_layer_lists_are_checked(zf):
    kv = zf.KvManager(num_pages=4, num_raw_slots=4, page_size=P, max_requests=1, max_pages_per_req=4, num_layers=2)
    kv.admit(0, 16)
    with pytest.raises(ValueError):
        kv.reclaim([0], [[False]])                     # one row per layer
    with pytest.raises(zf.ZfError):
        zf.KvManager(num_pages=4, num_raw_slots=1, page_size=P, max_requests=1, max_pages_per_req=4, num_layers=2)


def test_plan_pages_counts_compressed_and_dense_storage(zf):
    # one layer, 8 kv heads, 16-token pages: a dense page is 2 x 8 x 4 x 1024 B; a page id costs
    # 2 x 8 x 4 x 784 B of slots + 8 directory entries
    dense_page = 2 * 8 * 4 * 1024
    comp_page = 2 * 8 * 4 * 784 + 8 * 4
    pages, dense = zf.kv_plan_pages(1000 * dense_page, 8, 16, 100)
    assert dense == 1000
    assert pages == (1000 - 100) * dense_page // comp_page
    assert 1.15 < pages / (dense - 100) < 1.31


@pytest.mark.parametrize("layers", [1, 3])
def test_random_workload_against_a_model(zf, layers):
    """Random admits, appends, reclaims and releases; after every call the manager's exported
    table, lengths and counts match a plain model of the rules and no id or slot is held twice."""
    rng = random.Random(5 + layers)
    NP, NR, R, MP = 60, 24 * layers, 6, 12
    kv = zf.KvManager(num_pages=NP, num_raw_slots=NR, page_size=P, max_requests=R, max_pages_per_req=MP,
                      num_layers=layers)
    model = {}                 # req -> dict(len, pages, tail_raw: per-layer slots or None)
    raw_kept = {}              # pid -> {layer: slot}, full pages left raw in some layers
    pending = {}               # pid -> per-layer slots

    def held_slots():
        s = [x for m in model.values() if m["tail_raw"] is not None for x in m["tail_raw"]]
        return s + [x for v in pending.values() for x in v] + [x for v in raw_kept.values() for x in v.values()]

    def cols(rs, i):
        return [rs[l][i] for l in range(layers)]

    for step in range(600):
        op = rng.random()
        free_ids = NP - sum(len(m["pages"]) for m in model.values())
        free_raw = NR - len(held_slots())
        openable = min(free_ids, free_raw // layers)
        if op < 0.2 and len(model) < R:
            req = rng.choice([q for q in range(R) if q not in model])
            length = rng.randint(0, 70)
            need = -(-length // P)
            if need > MP:
                continue
            if need > openable:
                with pytest.raises(zf.ZfError, match="page ids or raw slots"):
                    kv.admit(req, length)
                continue
            ids, nv, rs = kv.admit(req, length)
            assert nv == [min(P, length - i * P) for i in range(need)] and len(rs) == layers
            m = {"len": length, "pages": ids, "tail_raw": None}
            for i, (pid, fill) in enumerate(zip(ids, nv)):
                if fill == P:
                    pending[pid] = cols(rs, i)
                else:
                    m["tail_raw"] = cols(rs, i)
            model[req] = m
        elif op < 0.7 and model:
            reqs = rng.sample(sorted(model), rng.randint(1, len(model)))
            opening = [q for q in reqs if model[q]["len"] % P == 0]
            if any(-(-model[q]["len"] // P) + 1 > MP for q in opening):
                continue
            if len(opening) > openable:
                with pytest.raises(zf.ZfError, match="page ids or raw slots"):
                    kv.append(reqs)
                continue
            ids, nv, rs = kv.append(reqs)
            for i, (q, pid, fill) in enumerate(zip(reqs, ids, nv)):
                m = model[q]
                slots = cols(rs, i)
                if m["len"] % P == 0:
                    assert pid not in m["pages"]
                    m["pages"].append(pid)
                else:
                    assert slots == m["tail_raw"] and pid == m["pages"][-1]
                m["len"] += 1
                assert fill == m["len"] - (len(m["pages"]) - 1) * P
                if fill == P:
                    pending[pid] = slots
                    m["tail_raw"] = None
                else:
                    m["tail_raw"] = slots
        elif op < 0.85 and pending:
            ids, slots = kv.pending()
            assert {pid: cols(slots, i) for i, pid in enumerate(ids)} == pending
            pick = rng.sample(ids, rng.randint(1, len(ids)))
            kept = [[rng.random() < 0.1 for _ in pick] for _ in range(layers)]
            kv.reclaim(pick, kept)
            for i, pid in enumerate(pick):
                slots_p = pending.pop(pid)
                keep = {l: slots_p[l] for l in range(layers) if kept[l][i]}
                if keep:
                    raw_kept[pid] = keep
        elif model:
            req = rng.choice(sorted(model))
            kv.release(req)
            for pid in model.pop(req)["pages"]:
                pending.pop(pid, None)
                raw_kept.pop(pid, None)
        # compare
        table, lens = kv.export()
        for q in range(R):
            if q in model:
                m = model[q]
                assert lens[q] == m["len"]
                row = table[q].tolist()
                assert row[: len(m["pages"])] == m["pages"] and all(x == -1 for x in row[len(m["pages"]):])
            else:
                assert lens[q] == 0 and (table[q] == -1).all()
        all_ids = [p for m in model.values() for p in m["pages"]]
        assert len(all_ids) == len(set(all_ids))
        slots = held_slots()
        assert len(slots) == len(set(slots)) and all(0 <= s < NR for s in slots)
        st = kv.stats()
        assert st["free_pages"] == NP - len(all_ids) and st["free_raw_slots"] == NR - len(slots)
        assert st["pending_pages"] == len(pending) and st["raw_full_pages"] == len(raw_kept)
        assert st["raw_full_slots"] == sum(len(v) for v in raw_kept.values())
        assert st["new_page_capacity"] == min(NP - len(all_ids), (NR - len(slots)) // layers)
        assert st["tokens"] == sum(m["len"] for m in model.values())


def test_serving_loop_on_the_oracle_with_one_raw_pool(zf):
    """The manager's protocol end to end on the oracle's caches: two layers whose caches share one
    raw pool (the same arrays), prompts written with encode_pages, decode steps with append_tokens,
    raw slots reclaimed layer by layer from the directories after every step, a request released
    and another admitted mid-way.  Layer 1's keys carry blocks that cannot be encoded (eight tiny
    values in a 512-value block), so some pages stay raw there only.  After every step each
    layer's pages hold every request's tokens bit for bit — a slot handed from one layer to the
    other never overwrites live data."""
    import numpy as np
    from oracle import zf_oracle as O

    Hkv, NL, max_len = 2, 2, 120
    rng = np.random.default_rng(3)

    def stream(spiky):
        x = rng.standard_normal((max_len, Hkv, 128)).astype(np.float32)
        if spiky:
            x[7::24, 0, 5:13] *= 2.0 ** -30
        return ((x.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)

    sk = [[stream(l == 1) for _ in range(4)] for l in range(NL)]
    sv = [[stream(False) for _ in range(4)] for l in range(NL)]
    kv = zf.KvManager(num_pages=30, num_raw_slots=14, page_size=P, max_requests=4, max_pages_per_req=8, num_layers=NL)
    caches = [O.Cache(num_pages=30, num_kv_heads=Hkv, page_size=P, num_raw=14) for _ in range(NL)]
    caches[1].k_raw, caches[1].v_raw = caches[0].k_raw, caches[0].v_raw
    stream_of = {}

    def reclaim():
        ids, _ = kv.pending()
        if ids:
            kv.reclaim(ids, [[bool((c.dir[pid] >= 0).any()) for pid in ids] for c in caches])

    def admit(req, length):
        stream_of[req] = req
        ids, nv, rs = kv.admit(req, length)
        for l in range(NL):
            src_k = np.zeros((len(ids), Hkv, P, 128), np.uint16)
            src_v = np.zeros_like(src_k)
            for j, fill in enumerate(nv):
                src_k[j, :, :fill] = sk[l][req][j * P:j * P + fill].transpose(1, 0, 2)
                src_v[j, :, :fill] = sv[l][req][j * P:j * P + fill].transpose(1, 0, 2)
            O.encode_pages(caches[l], src_k, src_v, ids, nv, rs[l])
        reclaim()

    def check():
        table, lens = kv.export()
        for l in range(NL):
            for req, s in stream_of.items():
                L = int(lens[req])
                K, V = O.gather_sequence(caches[l], table[req].numpy(), L)
                assert (K == sk[l][s][:L]).all() and (V == sv[l][s][:L]).all(), (l, req)
            assert caches[l].status == 0

    for req, length in ((0, 37), (1, 16), (2, 50)):
        admit(req, length)
    check()
    for step in range(30):
        if step == 12:
            kv.release(1)
            del stream_of[1]
            admit(3, 21)
        reqs = sorted(stream_of)
        ids, nv, rs = kv.append(reqs)
        lens = kv.export()[1]
        for l in range(NL):
            k_tok = np.stack([sk[l][stream_of[q]][int(lens[q]) - 1] for q in reqs])
            v_tok = np.stack([sv[l][stream_of[q]][int(lens[q]) - 1] for q in reqs])
            O.append_tokens(caches[l], k_tok, v_tok, ids, [f - 1 for f in nv], rs[l])
        reclaim()
        check()
    st = kv.stats()
    assert st["pending_pages"] == 0 and st["raw_full_pages"] > 0
    assert st["raw_full_slots"] == st["raw_full_pages"]          # kept in layer 1 only
