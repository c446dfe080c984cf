"""The prompt-cache index (tfl_prefix_store_*) on the host: longest common
token prefix, ties to the entry put last, capacity, removal.  The store never
touches a cache, so stand-in handles serve here."""
import ctypes

import pytest

from gqa_decoder_forward_gb300 import tfl


class _FakeKV:
    def __init__(self, addr):
        self.handle = ctypes.c_void_p(addr)


@pytest.fixture
def store():
    return tfl.PrefixStore(3)


def test_longest_prefix_wins(store):
    a, b = _FakeKV(0x1000), _FakeKV(0x2000)
    store.put([1, 2, 3, 4, 5], a)
    store.put([1, 2, 9], b)
    kv, n = store.match([1, 2, 3, 4, 7, 8])
    assert kv is a and n == 4
    kv, n = store.match([1, 2, 9, 9])
    assert kv is b and n == 3
    kv, n = store.match([1, 2])
    assert kv is b and n == 2            # tie at 2: the entry put last
    kv, n = store.match([5, 1, 2])
    assert kv is None and n == 0
    kv, n = store.match([])
    assert kv is None and n == 0


def test_capacity_and_remove(store):
    kvs = [_FakeKV(0x100 * (i + 1)) for i in range(4)]
    for i in range(3):
        store.put([i, i + 1], kvs[i])
    assert len(store) == 3
    with pytest.raises(tfl.TflError) as e:
        store.put([9], kvs[3])
    assert e.value.code == tfl.TFL_E_CAPACITY
    store.remove(kvs[1])
    assert len(store) == 2
    assert store.match([1, 2])[0] is None
    store.put([9], kvs[3])
    assert store.match([9, 9]) == (kvs[3], 1)


def test_bad_arguments(store):
    with pytest.raises(tfl.TflError):
        store.put([], _FakeKV(0x10))
    with pytest.raises(tfl.TflError):
        tfl.PrefixStore(0)
