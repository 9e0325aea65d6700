"""clo_wait_ready / clo_signal_ready on the GPU: the GPU-centric data-ready
synchronisation of CLO (a kernel already on the stream polls a flag that a
host thread publishes).  Every wait here is bounded (a few ms to 2 s): the
flag that nothing sets makes the wait run out, and the test checks the
status it leaves and that the stream and context still work afterwards."""
import threading
import time

import numpy as np
import pytest
import torch

import offloaded_kv_decode_gb300 as clo
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _flag(value=0):
    f = torch.zeros(1, dtype=torch.int32).pin_memory()
    f.view(torch.uint8)[:4] = torch.tensor(np.array([value], dtype=np.uint32).view(np.uint8))
    return f


def _timed(fn):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    return a, b


def test_value_already_there_passes_at_once():
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    f = _flag(5)
    for expected in (5, 3, 0xFFFFFFF0):  # equal, older, and older across the wrap of 2^32
        a, b = _timed(lambda: clo.clo_wait_ready(f, expected, 2_000_000, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert a.elapsed_time(b) < 50.0


def _load_copy_kernel():
    """One copy launch, so the copy queued behind a wait below is not its
    kernel's first launch (under lazy module loading a first launch can wait
    for the device to go idle, i.e. for the wait)."""
    src = torch.ones(16, dtype=torch.int32).pin_memory()
    dst = torch.zeros(16, dtype=torch.int32, device=dev())
    clo.clo_copy_async([(dst, src)])
    torch.cuda.synchronize()


def test_wait_ends_when_the_host_signals_and_sees_the_data():
    """The host thread fills a pinned buffer, then publishes the flag; the GPU
    wait, then a copy of that buffer queued behind it, see the new data."""
    _load_copy_kernel()
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    f = _flag(0)
    host = torch.zeros(1 << 20, dtype=torch.int32).pin_memory()
    dst = torch.full((1 << 20,), -1, dtype=torch.int32, device=d)
    payload = torch.arange(1 << 20, dtype=torch.int32) * 7 + 3

    def producer():
        time.sleep(0.03)
        host.copy_(payload)
        clo.clo_signal_ready(f, 1)

    t = threading.Thread(target=producer)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    clo.clo_wait_ready(f, 1, 2_000_000, err)
    clo.clo_copy_async([(dst, host)])
    b.record()
    t.start()  # the launches are queued before the data exists
    t.join()   # (joined before synchronising: the host thread must not need the GIL then)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert a.elapsed_time(b) >= 20.0
    assert torch.equal(dst.cpu(), payload)


def test_sequence_numbers_wrap_around():
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    f = _flag(0xFFFFFFF0)
    t = threading.Thread(target=lambda: (time.sleep(0.01), clo.clo_signal_ready(f, 2)))
    clo.clo_wait_ready(f, 0xFFFFFFF8, 2_000_000, err)
    t.start()
    t.join()
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_flag_never_set_times_out_and_the_context_stays_usable():
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    f = _flag(0)
    a, b = _timed(lambda: clo.clo_wait_ready(f, 1, 50_000, err))
    torch.cuda.synchronize()
    flag = int(err.item())
    assert flag & clo.FLAG_TIMEOUT
    assert clo.check_error_flag(flag) == clo.CLO_ERR_TIMEOUT
    assert 45.0 <= a.elapsed_time(b) < 1000.0
    # The stream and the library still work.
    src = torch.arange(4096, dtype=torch.int32).pin_memory()
    dst = torch.zeros(4096, dtype=torch.int32, device=d)
    clo.clo_copy_async([(dst, src)])
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)


def test_device_memory_flag():
    """A flag in device memory (set before the wait by an ordinary copy on the
    same stream) is accepted and read."""
    d = dev()
    err = torch.zeros(1, dtype=torch.int32, device=d)
    f = torch.zeros(1, dtype=torch.int32, device=d)
    f.fill_(9)
    clo.clo_wait_ready(f, 9, 100_000, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_rejects_pageable_host_memory():
    f = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(clo.CloError):
        clo.clo_wait_ready(f, 1, 1000)
