"""The binding refuses tensors and streams of another device before any
launch.  The library launches on the calling thread's current CUDA device
and dereferences every pointer there; a tensor of another GPU would make a
kernel touch memory that device cannot address.  The rule itself is host
logic, checked here without a GPU."""

import pytest
import torch

from replication_token_warp_gb300 import kvpub


def test_current_device_passes():
    kvpub.check_devices([torch.device("cuda", 0)] * 3, 0)
    kvpub.check_devices([torch.device("cuda", 3)], 3)


@pytest.mark.parametrize("dev", [torch.device("cuda", 1), torch.device("cpu"),
                                 torch.device("meta")])
def test_other_devices_are_refused(dev):
    with pytest.raises(ValueError, match="current CUDA device cuda:0"):
        kvpub.check_devices([torch.device("cuda", 0), dev], 0)


def test_device_indices_are_accepted_too():
    kvpub.check_devices([0, 0, torch.device("cuda", 0)], 0)
    with pytest.raises(ValueError, match="cuda:2 is not the current CUDA device cuda:0"):
        kvpub.check_devices([0, 2], 0)
    with pytest.raises(ValueError, match="cpu is not the current CUDA device"):
        kvpub.check_devices([-1], 0)


def test_store_arguments_are_checked_against_the_current_device(monkeypatch):
    """_store_args compares every tensor's device with the current one; on a
    machine without a GPU this runs with stand-in tensors whose devices are
    set by hand."""

    class FakeTensor:
        def __init__(self, device, dtype, shape):
            self.device = torch.device(device)
            self.dtype, self.shape = dtype, shape
            self._stride = (shape[1], 1) if len(shape) == 2 else (1,)
            self.is_cuda = self.device.type == "cuda"

        def get_device(self):
            return self.device.index if self.device.type == "cuda" else -1

        def dim(self):
            return len(self.shape)

        def stride(self, i=None):
            return self._stride if i is None else self._stride[i]

        def is_contiguous(self):
            return True

        def data_ptr(self):
            return 4096

        def numel(self):
            n = 1
            for x in self.shape:
                n *= x
            return n

    monkeypatch.setattr(kvpub, "_current_device", lambda: 0)
    T, nb = 4, 2

    def args(cache_dev):
        bf = torch.bfloat16
        return (FakeTensor("cuda:0", bf, (T, 512)), FakeTensor("cuda:0", bf, (T, 64)),
                FakeTensor("cuda:0", bf, (T, 128)), FakeTensor("cuda:0", torch.int64, (T,)),
                [FakeTensor(cache_dev, torch.uint8, (nb * 64 * 656,))],
                [FakeTensor("cuda:0", torch.uint8, (nb * 8448,))], nb, None)

    out = kvpub._store_args(*args("cuda:0"))
    assert out[7] == T and out[10] == 1
    with pytest.raises(ValueError, match="cuda:1 is not the current CUDA device"):
        kvpub._store_args(*args("cuda:1"))
