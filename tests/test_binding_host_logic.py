"""The binding's argument checks that run before any CUDA call (CPU only):
a call on device tensors refuses host output tensors, a host gamax it would
have to write, and a residual that is not on x's device (its kernels would be
handed host pointers, or the in-place update would land in a staged copy);
given tensors of the wrong dtype or size are refused before the kernels could
read or write past them."""
import pytest
import torch

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


def test_device_call_refuses_host_outputs():
    with pytest.raises(ValueError):
        nv._out_buf((4, 8), torch.uint8, torch.empty((4, 8), dtype=torch.uint8), torch.device("cuda", 0), False)


def test_device_call_refuses_foreign_residual():
    with pytest.raises(ValueError):
        nv._dev_residual(torch.zeros((4, 16)), torch.device("cuda", 0))
    assert nv._dev_residual(None, torch.device("cuda", 0)) is None


DEV = torch.device("cuda", 0)


def test_device_call_refuses_a_host_gamax_to_write():
    for mode in (nv.GAMAX_TENSOR, nv.GAMAX_ROW):
        with pytest.raises(ValueError):
            nv._gamax_buffer(mode, torch.zeros(64), 64, DEV, host=False)


def test_host_call_checks_a_given_host_gamax():
    with pytest.raises(ValueError):                     # wrong dtype
        nv._gamax_buffer(nv.GAMAX_TENSOR, torch.zeros(1, dtype=torch.float64), 64, DEV, host=True)
    with pytest.raises(ValueError):                     # 'row' needs M floats
        nv._gamax_buffer(nv.GAMAX_ROW, torch.zeros(8), 64, DEV, host=True)
    with pytest.raises(ValueError):                     # a written amax needs a tensor
        nv._gamax_buffer(nv.GAMAX_TENSOR, 3.0, 64, DEV, host=True)


def test_host_call_checks_the_residual():
    nv._host_residual(None, 4, 16)
    nv._host_residual(torch.zeros(4, 16), 4, 16)
    with pytest.raises(ValueError):
        nv._host_residual(torch.zeros(4, 16, dtype=torch.bfloat16), 4, 16)
    with pytest.raises(ValueError):
        nv._host_residual(torch.zeros(4, 8), 4, 16)


def test_host_call_checks_given_host_outputs():
    with pytest.raises(ValueError):
        nv._out_buf((4, 8), torch.uint8, torch.empty((4, 8), dtype=torch.int8), DEV, True, "codes")
    with pytest.raises(ValueError):
        nv._out_buf((4, 8), torch.uint8, torch.empty((4, 4), dtype=torch.uint8), DEV, True, "codes")


def test_device_checks_reject_wrong_tensors_before_any_cuda_call():
    t = torch.zeros(4, 16)
    with pytest.raises(ValueError):                     # not on the call's device
        nv._check_dev(t, "residual", torch.float32, 64, DEV)


def test_pipelined_row_chunks_cover_the_rows_in_whole_tiles():
    """The pipelined host path's chunks: at most eight, contiguous, covering
    every row once, each starting on a multiple of 16 rows (whole 16x16
    tiles, and the chunk's row_offset keeps the stochastic-rounding index)."""
    for M in (256, 300, 1040, 4096, 14336, 16384, 16400):
        ch = nv._row_chunks(M)
        assert 1 <= len(ch) <= 8
        assert ch[0][0] == 0 and ch[-1][1] == M
        for (a, b), (c, _) in zip(ch, ch[1:]):
            assert b == c
        for a, b in ch:
            assert a % 16 == 0 and b > a


class _Event:
    def __init__(self, done):
        self.done = done

    def query(self):
        return self.done


class _Stream:
    def __init__(self):
        self.waited = []

    def wait_event(self, ev):
        self.waited.append(ev)


def test_non_blocking_reads_wait_for_overlapping_pending_writes():
    """A host tensor that an unfinished non-blocking call writes is read by a
    later call only after that write's event: the reading stream waits for
    exactly the events whose host byte ranges overlap the tensors it reads
    (views of the same storage included); finished writes are dropped."""
    dev = torch.device("cuda", 7)                       # a key only: nothing runs on it
    a, b, c = torch.zeros(64), torch.zeros(64), torch.zeros(16)
    view = a[32:]
    e1, e2, e3 = _Event(False), _Event(False), _Event(True)
    nv._pending.pop(dev, None)
    try:
        nv._add_pending(dev, [a], e1)
        nv._add_pending(dev, [b], e2)
        nv._add_pending(dev, [c], e3)
        st = _Stream()
        nv._wait_pending(dev, st, [view])
        assert st.waited == [e1]
        st = _Stream()
        nv._wait_pending(dev, st, [c, torch.zeros(8)])
        assert st.waited == []                          # c's write finished; a new tensor has none
        assert [p[2] for p in nv._pending[dev]] == [e1, e2]
        e1.done = e2.done = True
        nv._wait_pending(dev, _Stream(), [a])
        assert nv._pending[dev] == []
    finally:
        nv._pending.pop(dev, None)
    assert nv._ranges_overlap((0, 10), (9, 20)) and not nv._ranges_overlap((0, 10), (10, 20))


def test_non_blocking_host_calls_refuse_a_stream():
    with pytest.raises(ValueError):
        nv._non_blocking_stream(True, object())
    nv._non_blocking_stream(True, None)
    nv._non_blocking_stream(False, object())
    with pytest.raises(ValueError):
        nv._non_blocking_refused(True)


def test_product_and_probe_operands_must_be_device_tensors():
    """nvfp4_mm and the diagnostics hand their tensors' pointers to kernels
    as they are: host tensors are refused before any CUDA call."""
    z = torch.zeros(128 * 64, dtype=torch.uint8)
    with pytest.raises(ValueError):
        nv._check_mm_args(z, z, z, z, 128, 128, 128, None, None, None, nv.BF16)
    with pytest.raises(ValueError):
        nv._check_probe_inputs((torch.ones(4), torch.float32, "a"))
    with pytest.raises(ValueError):                     # wrong dtype is refused before the device test
        nv._check_probe_inputs((torch.ones(4, dtype=torch.int32), torch.float32, "v"))



def test_error_feedback_keeps_one_residual_per_name():
    from nvfp4_block_quantization_quantize_gb300.error_feedback import ErrorFeedback
    ef = ErrorFeedback(stochastic=False)
    w = torch.ones(4, 16)
    r = ef.residual("a", w)
    assert r.dtype == torch.float32 and r.shape == w.shape and not r.any()
    r += 1.0
    assert ef.residual("a", w) is r                      # carried, not re-created
    with pytest.raises(ValueError):                     # another shape: refused, not reset
        ef.residual("a", torch.ones(4, 32))
    ef.residual("b", torch.ones(2, 16))
    assert sorted(ef.names()) == ["a", "b"]
    ef.reset("a")
    assert not ef.residual("a", w).any()
    ef.reset()
    assert ef.names() == []
