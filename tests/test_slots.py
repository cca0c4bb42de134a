"""Host slot table of the shared KV cache (no GPU): lowest free row on
admission, rows freed on stop / length / cancel, one decode step packs the
[3, capacity] token/position/row metadata and advances the rows."""
import pytest
import torch

import kv_cached_gqa_rope_gb300 as kv


def code_of(fn, *a):
    with pytest.raises(kv.KvgqaError) as e:
        fn(*a)
    return e.value.code


def test_lowest_free_row_and_reuse():
    t = kv.SlotTable(4, 32)
    assert [t.admit(r, 1) for r in (100, 101, 102, 103)] == [0, 1, 2, 3]
    assert code_of(t.admit, 104, 1) == "EFULL"
    t.release(102, kv.STOP)
    t.release(100, kv.CANCEL)
    assert t.admit(105, 2) == 0          # lowest free row first
    assert t.admit(106, 2) == 2
    assert t.admit(105, 9) == 0          # an admitted request keeps its row
    q = t.query()
    assert q["active"] == 4 and q["free"] == 0
    assert q["released"] == {"stop": 1, "length": 0, "cancel": 1}


def test_bad_arguments():
    with pytest.raises(kv.KvgqaError):
        kv.SlotTable(0, 8)
    t = kv.SlotTable(2, 8)
    assert code_of(t.admit, 1, 9) == "EINVAL"     # prompt longer than a row
    assert code_of(t.admit, 1, -1) == "EINVAL"
    assert code_of(t.release, 7, kv.STOP) == "EINVAL"
    t.admit(1, 0)
    assert code_of(t.release, 1, 5) == "EINVAL"


def test_step_packs_metadata_and_advances():
    t = kv.SlotTable(3, 8)
    t.admit(11, 4)
    t.admit(22, 0)
    meta = torch.full((3, 6), -7, dtype=torch.int32)
    A, fin = t.step([22, 11], [501, 502], meta)
    assert A == 2 and not fin.any()
    assert meta[:, :2].tolist() == [[501, 502], [0, 4], [1, 0]]
    assert meta[:, 2:].eq(-7).all()                  # entries past A untouched
    A, _ = t.step([11, 22], [7, 8], meta)
    assert meta[:, :2].tolist() == [[7, 8], [5, 1], [0, 1]]


def test_step_rejects_without_changing_anything():
    t = kv.SlotTable(2, 8)
    t.admit(1, 3)
    meta = torch.zeros(3, 4, dtype=torch.int32)
    for reqs in ([1, 9], [1, 1]):                    # unknown, repeated
        with pytest.raises(kv.KvgqaError) as e:
            t.step(reqs, [0] * len(reqs), meta)
        assert e.value.code == "EINVAL"
    A, _ = t.step([1], [0], meta)
    assert meta[1, 0] == 3                            # the failed steps did not advance the row
    with pytest.raises(ValueError):
        t.step([1], [0], torch.zeros(3, 4, dtype=torch.int64))
    with pytest.raises(kv.KvgqaError):
        t.step([1, 1, 1, 1, 1], [0] * 5, meta)       # more entries than capacity


def test_length_release():
    t = kv.SlotTable(2, 4)
    t.admit(5, 2)
    t.admit(6, 0)
    meta = torch.zeros(3, 2, dtype=torch.int32)
    _, fin = t.step([5, 6], [0, 0], meta)            # request 5: positions 2 -> length 3
    assert not fin.any()
    _, fin = t.step([5, 6], [0, 0], meta)            # request 5 writes position 3: row full
    assert fin.tolist() == [True, False]
    assert meta[1].tolist() == [3, 1]
    assert t.query()["released"]["length"] == 1
    assert t.admit(7, 1) == 0                         # the freed row is reused
