"""The Python binding's checks of the buffers a step writes or reads (no GPU):
the library takes raw device pointers and cannot see sizes, so a buffer that is
too small, of the wrong dtype or device, or strided must be refused before
anything is launched."""
import pytest
import torch

from decode_megakernel_persistent_gb300 import ll


class FakeCuda:
    """Stands in for a CUDA tensor (none exists on a CPU-only machine)."""

    def __init__(self, n, dtype=torch.float32, device="cuda:0", contiguous=True):
        self.is_cuda = True
        self.dtype = dtype
        self.device = torch.device(device)
        self._n = n
        self._c = contiguous

    def numel(self):
        return self._n

    def is_contiguous(self):
        return self._c


DEV = torch.device("cuda:0")


def refused(t, dtype=torch.float32, n=10, optional=True):
    with pytest.raises(ll.LLError) as e:
        ll._need(t, "buf", dtype, n, DEV, optional)
    assert e.value.code == ll.LL_ERR_ARG
    return str(e.value)


def test_accepts_a_fitting_buffer_and_optional_none():
    ll._need(FakeCuda(10), "buf", torch.float32, 10, DEV)
    ll._need(FakeCuda(11), "buf", torch.float32, 10, DEV)
    ll._need(None, "buf", torch.float32, 10, DEV)


def test_refuses_bad_buffers():
    assert "required" in refused(None, optional=False)
    assert "CUDA" in refused(torch.zeros(10))                       # host tensor
    assert "int32" in refused(FakeCuda(10), dtype=torch.int32)       # wrong dtype
    assert "cuda:1" in refused(FakeCuda(10, device="cuda:1"))        # other device
    assert "contiguous" in refused(FakeCuda(10, contiguous=False))
    assert "needs 10" in refused(FakeCuda(9))                        # one element short
