"""The update calls' work items, from the library itself on the host (no GPU): how a tensor list is cut into slices
of large tensors and packs of small ones, the pack table the kernels search, and the order the kernels take the
items in. Every octet (8 elements) of every tensor must belong to exactly one item."""
import ctypes

import numpy as np
import pytest

import clip_tensor_adamw_gb300 as mica

OK, NULL, COUNT = 0, 1, 2


def octs(n):
    return (n + 7) // 8


def check_items(sizes, vec, io):
    items, pack, used = mica.mica_work_items(sizes, vec, item_octs=io)
    if io:
        assert used == io
    io = used
    small, cap = min(512, io), min(1536, 3 * io)
    covered = [np.zeros(octs(n), np.int32) for n in sizes]
    packs = []
    for t, c, o0 in items:
        assert 0 <= t and c >= 1 and t + c <= len(sizes)
        if c == 1:  # a slice of tensor t (or a small tensor alone)
            no = octs(sizes[t])
            assert 0 <= o0 < no and o0 % io == 0, (t, o0, no)
            covered[t][o0:min(o0 + io, no)] += 1
        else:  # a pack: tensors t .. t+c-1 whole, its row of the pack table at pack[o0]
            members = range(t, t + c)
            assert all(octs(sizes[k]) <= small for k in members)
            assert sum(octs(sizes[k]) for k in members) <= cap
            pre_w = pack[o0:o0 + c + 1]
            pre_e = pack[o0 + c + 1:o0 + 2 * c + 2]
            whole = [sizes[k] // 8 if vec[k] else 0 for k in members]
            other = [octs(sizes[k]) - w for k, w in zip(members, whole)]
            assert pre_w == [int(x) for x in np.concatenate([[0], np.cumsum(whole)])]
            assert pre_e == [int(x) for x in np.concatenate([[0], np.cumsum(other)])]
            for k in members:
                covered[k] += 1
            packs.append(t)
    for k, cov in enumerate(covered):
        assert (cov == 1).all(), (k, sizes[k], cov)
    # the kernels take items from the end of the array: packs first, each followed by a slice, while both last;
    # the slices from the end of the list backwards
    taken = items[::-1]
    kinds = ["P" if c > 1 else "S" for _, c, _ in taken]
    np_, ns = kinds.count("P"), kinds.count("S")
    if np_ and ns:
        if np_ <= ns:
            assert kinds[:2 * np_] == ["P", "S"] * np_ and set(kinds[2 * np_:]) <= {"S"}
        else:  # more packs than slices: the packs spread evenly over the slices
            pos = [i for i, k in enumerate(kinds) if k == "S"]
            for i, p in enumerate(pos):
                before = p - i
                assert i * np_ / ns <= before <= i * np_ / ns + 1, (i, before, np_, ns)
    slices = [(t, o0) for t, c, o0 in taken if c == 1]
    assert slices == sorted(slices, reverse=True)
    pack_starts = [t for t, c, _ in taken if c > 1]
    assert pack_starts == sorted(pack_starts, reverse=True)
    return items, pack, io


@pytest.mark.parametrize("io", [16, 64, 512, 0])
@pytest.mark.parametrize("seed", range(6))
def test_every_octet_in_exactly_one_item(seed, io):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 400))
    kind = seed % 3
    if kind == 0:
        sizes = [int(x) for x in np.floor(np.exp(rng.uniform(np.log(1), np.log(300_000), T)))]
    elif kind == 1:
        sizes = [int(x) for x in rng.integers(0, 40, T)]
    else:
        sizes = [int(x) for x in np.floor(np.exp(rng.uniform(np.log(64), np.log(4096), T)))] + [768 * 3072] * 3
    vec = [bool(b) for b in rng.random(len(sizes)) < 0.8]
    check_items(sizes, vec, io)


def test_loss_scaled_list_shape():
    """10,000 small tensors then 12 large ones: all small tensors in packs (at most 1,024 octets each), the large
    ones in 512-octet slices, and the packs taken first, each beside a slice."""
    rng = np.random.default_rng(0)
    sizes = [int(x) for x in np.floor(np.exp(rng.uniform(np.log(64), np.log(4096), 10_000)))] + [768 * 3072] * 12
    items, pack, io = check_items(sizes, [True] * len(sizes), 0)
    assert io == 512
    slices = [it for it in items if it[1] == 1]
    packs = [it for it in items if it[1] > 1]
    assert len(slices) == 12 * (768 * 3072 // 8 // 512)
    assert sum(c for _, c, _ in packs) == 10_000


def test_many_tiny_tensors_and_empty_ones():
    sizes = ([0] * 5 + list(range(10)) * 3000 + [0] * 5)
    check_items(sizes, [True] * len(sizes), 0)
    check_items(sizes, [k % 2 == 0 for k in range(len(sizes))], 16)


def test_item_size_follows_the_list(monkeypatch):
    """With no size given, 512 octets per slice (AdamW, float32 moments), halved down to 128 while the list would
    give fewer than 16 items per SM."""
    monkeypatch.delenv("MICA_ITEM_OCTS", raising=False)
    assert mica.mica_work_items([50_000_000])[2] == 512
    assert mica.mica_work_items([1_000_000])[2] == 128
    assert mica.mica_work_items([8 * 512 * 152 * 16])[2] == 512
    assert mica.mica_work_items([8 * 512 * 152 * 16 - 8])[2] == 256
    assert mica.mica_work_items([50_000_000], sms=10_000)[2] == 128


def test_work_items_host_validation():
    L = mica.lib()
    n = (ctypes.c_int64 * 2)(100_000, 5)  # 12,500 octets in 128-octet slices, then 5 elements alone
    v = (ctypes.c_int32 * 2)(1, 1)
    num, plen, used = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    args = lambda **kw: dict(dict(n=n, v=v, T=2, io=0, sms=152, items=None, mi=0, pack=None, mp=0,
                                  num=ctypes.byref(num), plen=ctypes.byref(plen), used=None), **kw)

    def call(**kw):
        a = args(**kw)
        return L.mica_work_items(a["n"], a["v"], a["T"], a["io"], a["sms"], a["items"], a["mi"], a["pack"], a["mp"],
                                 a["num"], a["plen"], a["used"])
    assert call() == OK and num.value == 12_500 // 128 + 1 + 1 and plen.value == 0
    assert call(num=None) == NULL
    assert call(n=None) == NULL
    assert call(mi=4) == NULL  # a capacity with no array
    assert call(T=-1) == COUNT
    for bad in (8, 17, 96, 1 << 21):
        assert call(io=bad) == COUNT, bad
    assert call(sms=0) == COUNT
    neg = (ctypes.c_int64 * 2)(100, -1)
    assert call(n=neg) == COUNT
    # a short output buffer: the full counts are still reported, only the capacity is written
    buf = (ctypes.c_int64 * 6)(*([-7] * 6))
    assert call(items=buf, mi=1) == OK and num.value == 12_500 // 128 + 2
    assert list(buf[3:]) == [-7, -7, -7] and list(buf[:3]) == [0, 1, 0]
    assert call(T=0, n=None, v=None) == OK and num.value == 0


def test_more_packs_than_slices():
    """167 packs of 30-element tensors (twelve a pack at 16-octet items, the last of eight) and one tensor of 40
    slices: the packs are spread evenly over the slices, and the launch still takes every octet once."""
    sizes = [30] * 2000 + [5000]
    items, _, _ = check_items(sizes, [True] * len(sizes), 16)
    kinds = ["P" if c > 1 else "S" for _, c, _ in items[::-1]]
    assert kinds.count("P") == 167 and kinds.count("S") == 40
    assert sorted(c for _, c, _ in items if c > 1) == [8] + [12] * 166
