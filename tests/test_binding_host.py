"""CPU tests of the Python binding's argument marshalling: the address of
every accepted buffer kind, and host int32 lengths passed through without a
copy when they already are int32 and C-contiguous (numpy or CPU tensor), and
converted otherwise."""
import numpy as np
import torch

import place_kv_cache_gb300 as ol


def test_addresses_of_every_buffer_kind():
    a = np.arange(8, dtype=np.int32)
    t = torch.arange(8, dtype=torch.int32)
    p = torch.nn.Parameter(torch.zeros(4))                 # a tensor subclass
    assert ol._ptr(None) is None
    assert ol._ptr(12345) == 12345
    assert ol._ptr(a) == a.ctypes.data
    assert ol._ptr(t) == t.data_ptr()
    assert ol._ptr(t) == t.data_ptr()                       # second call: the per-type fast path
    assert ol._ptr(p) == p.data_ptr()
    assert ol._ptr(t[2:]) == t.data_ptr() + 8               # views keep their own address


def test_int32_lengths_pass_through_without_a_copy():
    a = np.array([3, 5], np.int32)
    t = torch.tensor([3, 5], dtype=torch.int32)
    assert ol._host_i32(a) is a
    assert ol._host_i32(t) is t
    assert ol._host_i32(None) is None


def test_other_lengths_are_converted():
    for x in ([3, 5], (3, 5), np.array([3, 5], np.int64), torch.tensor([3, 5], dtype=torch.int64),
              np.array([[3, 5], [7, 9]], np.int32)[:, 0]):   # the last one is not contiguous
        y = ol._host_i32(x)
        assert isinstance(y, np.ndarray) and y.dtype == np.int32 and y.flags.c_contiguous
        assert list(y.reshape(-1)[:2]) in ([3, 5], [3, 7])
    strided = torch.tensor([[3, 5], [7, 9]], dtype=torch.int32)[:, 0]
    y = ol._host_i32(strided)
    assert y is not strided and list(np.asarray(y)) == [3, 7]
