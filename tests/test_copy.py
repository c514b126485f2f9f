"""dfa_copy: host <-> device and device <-> device copies through the SMs
(include/dfa.h).  Bytes must arrive unchanged for every size and alignment,
each copy is one counted launch of this library, and pointers the SMs cannot
reach (pageable host memory) or overlapping ranges are refused before
anything is launched."""
import ctypes

import pytest
import torch

from long_context_causal_gb300 import dfa

pytestmark = pytest.mark.gpu


def pattern(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 4096 + 3, 1_000_003, 256 << 20])
@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (0, 7), (5, 3)])
def test_bytes_arrive_unchanged_in_every_direction(nbytes, offsets):
    if nbytes == 256 << 20 and offsets != (0, 0):
        pytest.skip("one large aligned case is enough")
    so, do = offsets
    ref = pattern(nbytes, nbytes % 1000 + 7 * so + do)
    h_src = torch.empty(nbytes + so, dtype=torch.uint8).pin_memory()
    h_src[so:] = ref
    d_buf = torch.zeros(nbytes + do, dtype=torch.uint8, device="cuda")
    d_buf2 = torch.zeros(nbytes + so, dtype=torch.uint8, device="cuda")
    h_dst = torch.zeros(nbytes + do, dtype=torch.uint8).pin_memory()

    n0 = dfa.dfa_launch_count("copy")
    dfa.dfa_copy(d_buf[do:], h_src[so:])                 # host -> device
    dfa.dfa_copy(d_buf2[so:], d_buf[do:])                # device -> device
    dfa.dfa_copy(h_dst[do:], d_buf2[so:])                # device -> host
    torch.cuda.synchronize()
    dfa.dfa_check_errors()
    assert torch.equal(d_buf[do:].cpu(), ref)
    assert torch.equal(d_buf2[so:].cpu(), ref)
    assert torch.equal(h_dst[do:], ref)
    # nothing outside the destination ranges is written
    assert int(d_buf[:do].abs().sum()) == 0 and int(h_dst[:do].abs().sum()) == 0
    assert dfa.dfa_launch_count("copy") - n0 == 3


def test_a_zero_byte_copy_launches_nothing():
    a = torch.empty(0, dtype=torch.uint8, device="cuda")
    b = torch.empty(0, dtype=torch.uint8).pin_memory()
    n0 = dfa.dfa_launch_count("copy")
    dfa.dfa_copy(a, b)
    assert dfa.dfa_launch_count("copy") == n0


def test_memory_the_sms_cannot_reach_and_overlaps_are_refused():
    lib = dfa.library()
    dev = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(1 << 20, dtype=torch.uint8)
    n0 = dfa.dfa_launch_count("copy")
    with pytest.raises(ValueError, match="pinned"):
        dfa.dfa_copy(dev, pageable)
    # the C entry point itself checks the pointer kind
    st = lib.dfa_copy(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(pageable.data_ptr()),
                      ctypes.c_size_t(1 << 20), None)
    assert st == dfa.DFA_ERR_INVALID_ARG and "pageable" in dfa.dfa_last_error()
    st = lib.dfa_copy(ctypes.c_void_p(dev.data_ptr() + 16), ctypes.c_void_p(dev.data_ptr()),
                      ctypes.c_size_t(1024), None)
    assert st == dfa.DFA_ERR_INVALID_ARG and "overlap" in dfa.dfa_last_error()
    st = lib.dfa_copy(None, ctypes.c_void_p(dev.data_ptr()), ctypes.c_size_t(16), None)
    assert st == dfa.DFA_ERR_INVALID_ARG
    with pytest.raises(ValueError, match="byte counts"):
        dfa.dfa_copy(dev[:16], dev[16:48])
    assert dfa.dfa_launch_count("copy") == n0
