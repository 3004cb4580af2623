"""Host block manager (C++ in libpagedkv.so) against the plain-Python model, plus pins of
the model to what the pages state (CPU only)."""
import math
import random

import pytest
import torch

import workloads
from oracle.block_manager_model import BlockManagerModel, OutOfBlocks
from paged_kv_cache_310_gb300 import PagedKVError, _build
from paged_kv_cache_310_gb300.block_manager import BlockManager, waste_report


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def same_state(bm, model):
    ids = sorted(model.tables)
    if ids:
        mb = max(len(t) for t in model.tables.values()) or 1
        tables, lens = bm.block_tables(ids, max_blocks=mb)
        for i, s in enumerate(ids):
            want = model.tables[s] + [-1] * (mb - len(model.tables[s]))
            assert tables[i].tolist() == want
            assert int(lens[i]) == model.lens[s]
    assert bm.stats() == model.stats()


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(seed):
    rng = random.Random(310_500 + seed)
    bs = rng.choice([1, 4, 16])
    nb = rng.randint(8, 64)
    bm, model = BlockManager(nb, bs), BlockManagerModel(nb, bs)
    next_id = 0
    for _ in range(300):
        op = rng.random()
        live = sorted(model.tables)
        if op < 0.2 or not live:
            n = rng.randint(0, 3 * bs)
            try:
                model.add_sequence(next_id, n)
                ok = True
            except OutOfBlocks:
                ok = False
            if ok:
                bm.add_sequence(next_id, n)
            else:
                with pytest.raises(PagedKVError) as e:
                    bm.add_sequence(next_id, n)
                assert e.value.status == 7
            next_id += 1
        elif op < 0.35:
            parent = rng.choice(live)
            model.fork(parent, next_id)
            bm.fork(parent, next_id)
            next_id += 1
        elif op < 0.45 and (live or model.swapped):
            if model.swapped and rng.random() < 0.5:
                s = rng.choice(sorted(model.swapped))
                try:
                    want = model.swap_in(s)
                    ok = True
                except OutOfBlocks:
                    ok = False
                if ok:
                    assert bm.swap_in(s) == want
                else:
                    with pytest.raises(PagedKVError) as e:
                        bm.swap_in(s)
                    assert e.value.status == 7
            elif live:
                s = rng.choice(live)
                assert bm.swap_out(s) == model.swap_out(s)
        elif op < 0.85:
            seqs = rng.sample(live, rng.randint(1, len(live)))
            try:
                want_slots, want_pairs = model.append(seqs)
                ok = True
            except OutOfBlocks:
                ok = False
            if ok:
                slots, pairs = bm.append(seqs)
                assert slots.tolist() == want_slots
                assert [tuple(p) for p in pairs.tolist()] == want_pairs
            else:
                with pytest.raises(PagedKVError) as e:
                    bm.append(seqs)
                assert e.value.status == 7
        else:
            s = rng.choice(live)
            model.free_sequence(s)
            bm.free_sequence(s)
        same_state(bm, model)
        check_invariants(model)


def check_invariants(model):
    refs = [0] * model.num_blocks
    for t in model.tables.values():
        for b in t:
            refs[b] += 1
    assert refs == model.refs                                  # reference count = tables pointing at it
    assert sorted(model.free) == [b for b in range(model.num_blocks) if refs[b] == 0]
    for s, t in model.tables.items():
        assert len(t) == math.ceil(model.lens[s] / model.block_size)   # blocks only as tokens need them
    st = model.stats()
    assert st["stored_tokens"] <= st["allocated_slots"]
    # waste only in each block's unused tail: at most block_size - 1 rows per used block
    assert st["allocated_slots"] - st["stored_tokens"] <= st["used_blocks"] * (model.block_size - 1)


def test_shared_system_prompt_example():
    """Ten users share a 4,000-token system prompt stored once; their new tokens go to
    fresh 16-token blocks; a finished user's blocks go to the next request."""
    for M in (BlockManagerModel, BlockManager):
        m = M(400, 16)
        m.add_sequence(0, 4000)
        for u in range(1, 10):
            m.fork(0, u)
        st = m.stats()
        assert st["used_blocks"] == 250 and st["shared_blocks"] == 250
        slots, pairs = m.append(list(range(10)))
        assert len(pairs) == 0                                # 4000 = 250 x 16: nothing shared to copy
        slots = list(slots.tolist() if hasattr(slots, "tolist") else slots)
        assert len({s // 16 for s in slots}) == 10             # ten fresh blocks, one per user
        assert all(s % 16 == 0 for s in slots)
        st = m.stats()
        assert st["used_blocks"] == 260
        m.free_sequence(3)
        freed = slots[3] // 16
        assert m.stats()["used_blocks"] == 259                 # the shared prompt stays
        m.add_sequence(100, 5)
        t = m.block_tables([100], max_blocks=1)[0] if isinstance(m, BlockManager) else [m.tables[100]]
        first = int(t[0][0])
        assert first == freed                                  # reused on the very next request


def test_beam_search_copy_on_write_matches_the_workload():
    """Four beams forked from a prompt whose last block is partial: three copies, the
    fourth beam writes the original -- the reading behind the shared-prefix workload."""
    w = workloads.make_workload(4)
    prompts = w.meta["beam_prompts"]
    bm = BlockManager(4000, 16)
    total_pairs = 0
    for t, p in enumerate(prompts):
        root = 1000 * (t + 1)
        bm.add_sequence(root, p)
        beams = [root] + [root + k for k in range(1, 4)]
        for b in beams[1:]:
            bm.fork(root, b)
        slots, pairs = bm.append(beams)
        assert len(pairs) == 3
        assert len({int(s) // 16 for s in slots}) == 4        # every beam writes its own block
        total_pairs += len(pairs)
    assert total_pairs == w.cow_pairs.shape[0] == 24


def test_append_failure_changes_nothing():
    bm = BlockManager(3, 4)
    bm.add_sequence(1, 4)
    bm.add_sequence(2, 4)
    before = bm.stats()
    with pytest.raises(PagedKVError):
        bm.append([1, 2])              # both at a block boundary, only one free block
    assert bm.stats() == before
    with pytest.raises(PagedKVError):
        bm.append([1, 1])              # a sequence twice
    with pytest.raises(PagedKVError):
        bm.fork(7, 8)                  # unknown parent


def test_kv_waste_paged_vs_contiguous():
    """Waste stays in last-block tails (< 4 % here) while a max-length reservation
    wastes most of its memory for the same lengths."""
    g = torch.Generator().manual_seed(310_501)
    z = torch.randn(2000, generator=g, dtype=torch.float64)
    lens = [int(min(32768, max(1, round(math.exp(math.log(1024.0) + float(x)))))) for x in z]
    r = waste_report(lens, 16, 32768)
    assert r["paged_waste"] < 0.04
    assert r["allocated_slots"] - r["tokens"] <= len(lens) * 15
    assert r["contiguous_waste"] > 0.9
    # lengths uniform in [128, 2048] against a 2048-token reservation
    u = torch.randint(128, 2049, (2000,), generator=g).tolist()
    r2 = waste_report(u, 16, 2048)
    assert r2["paged_waste"] < 0.01 and 0.4 < r2["contiguous_waste"] < 0.5
