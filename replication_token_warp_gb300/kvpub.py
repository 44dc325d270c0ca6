"""ctypes binding of libkvpub (argument marshalling only).

Every operation runs in the CUDA library: these wrappers take torch CUDA
tensors, check their shapes (the C ABI cannot see sizes), pass raw device
pointers and the current torch stream, and raise ``KvpubError`` on a
non-zero status.  There is no fallback: if the library is not built, the
first call raises.

The library launches on the calling thread's current CUDA device, so every
tensor and stream passed here must live on that device; anything else is a
``ValueError`` before a launch (run the call under
``torch.cuda.device(tensor.device)``).

Names follow the C ABI in include/kvpub.h: ``store_mla_fp8`` (fused direct
publication into every replica), ``store_mla_bf16`` (the unquantised cache
variant), ``store_mla_fp8_publish`` (the same store
plus the device-epoch advance, one launch), ``gather_insert`` (the unfused
gather-then-insert path), ``epoch_advance`` and ``epoch_wait``.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

LATENT_DIM = 512
ROPE_DIM = 64
INDEXER_DIM = 128
BLOCK_SIZE = 64
MAIN_SLOT_BYTES = 656
INDEXER_BLOCK_BYTES = BLOCK_SIZE * 132
GATHER_ROW_BYTES = 1408
MAIN_SLOT_BYTES_BF16 = 1152
INDEXER_SLOT_BYTES_BF16 = 256
MAX_REPLICAS = 8
MAX_POLLS = 1 << 24
STATIC_GATHER_MAX_TOKENS = 4096

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "ALIGNMENT", 3: "TOO_MANY_REPLICAS", 4: "CUDA",
          5: "WORKSPACE"}


class KvpubError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"kvpub {STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_STORE_ARGS = [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
               ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.c_int, _i64, ctypes.c_int,
               _vp]

SIGNATURES = {
    "kvpub_store_mla_fp8": (_STORE_ARGS + [_vp], ctypes.c_int),
    "kvpub_store_mla_fp8_publish": (_STORE_ARGS + [_vp, _vp, _vp], ctypes.c_int),
    "kvpub_store_mla_bf16": (_STORE_ARGS + [_vp], ctypes.c_int),
    "kvpub_gather_workspace_bytes": ([_i64], ctypes.c_size_t),
    "kvpub_gather_insert": (_STORE_ARGS + [_vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "kvpub_gather_insert_noalloc": (_STORE_ARGS + [_vp], ctypes.c_int),
    "kvpub_epoch_advance": ([_vp, _vp], ctypes.c_int),
    "kvpub_epoch_wait": ([_vp, ctypes.c_uint64, ctypes.c_uint64, _vp, _vp], ctypes.c_int),
    "kvpub_last_error": ([], ctypes.c_char_p),
}


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with __graft_entry__.build() "
                    "(there is no fallback implementation)")
            handle = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
        return _lib


def last_error() -> str:
    return lib().kvpub_last_error().decode()


def check(status: int) -> None:
    if status != 0:
        raise KvpubError(status, last_error())


def check_devices(devices, current: int) -> None:
    """Raise ValueError unless every device in ``devices`` is CUDA device
    ``current``.  The library launches on the calling thread's current
    device and dereferences every pointer there, so a tensor (or stream) of
    another GPU would make a kernel touch memory it cannot address.  A
    device is a torch.device or a CUDA device index (``Tensor.get_device()``,
    -1 for a CPU tensor)."""
    for d in devices:
        if isinstance(d, int):
            if d == current:
                continue
            d = torch.device("cuda", d) if d >= 0 else torch.device("cpu")
        elif d.type == "cuda" and d.index == current:
            continue
        raise ValueError(f"{d} is not the current CUDA device cuda:{current}: call "
                         "under torch.cuda.device(...) of the tensors' device")


def _current_device() -> int:
    return torch.cuda.current_device()


def _stream_handle(stream, device: int) -> int:
    """The raw cudaStream_t to launch on: the current torch stream by
    default.  A torch.cuda.Stream must belong to ``device``, the device the
    call's tensors were checked against (a raw handle is passed as is)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        if stream.device_index != device:
            raise ValueError(f"stream of cuda:{stream.device_index} for tensors on the current "
                             f"CUDA device cuda:{device}: call under torch.cuda.device(...)")
        return stream.cuda_stream
    return int(stream)


def _rows(x: torch.Tensor, dim: int, T: int, name: str):
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D bf16 CUDA tensor")
    if x.stride(1) != 1 or x.shape[1] < dim or x.shape[0] < T:
        raise ValueError(f"{name}: expected [>= {T}, >= {dim}] rows with unit inner stride")
    return x.data_ptr(), x.stride(0)


def _ptr_array(ts):
    arr = (_vp * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


def _caches(main_caches, indexer_caches, num_blocks, main_slot=MAIN_SLOT_BYTES,
            indexer_block=INDEXER_BLOCK_BYTES):
    if len(main_caches) != len(indexer_caches):
        raise ValueError("need as many Indexer caches as Main caches")
    for c in list(main_caches) + list(indexer_caches):
        if not c.is_cuda or c.dtype != torch.uint8 or not c.is_contiguous():
            raise ValueError("caches are contiguous uint8 CUDA tensors")
    if num_blocks is None:
        num_blocks = main_caches[0].numel() // (BLOCK_SIZE * main_slot)
    for m, ix in zip(main_caches, indexer_caches):
        if (m.numel() < num_blocks * BLOCK_SIZE * main_slot
                or ix.numel() < num_blocks * indexer_block):
            raise ValueError(f"a cache is smaller than {num_blocks} blocks")
    return _ptr_array(main_caches), _ptr_array(indexer_caches), int(num_blocks)


def _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                num_blocks, invalid_count, bf16_cache=False):
    if slot_mapping.dtype != torch.int64 or slot_mapping.dim() != 1 or not slot_mapping.is_cuda:
        raise ValueError("slot_mapping: expected a 1-D int64 CUDA tensor")
    if not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous")
    T = slot_mapping.shape[0]
    lp, ls = _rows(kv_latent, LATENT_DIM, T, "kv_latent")
    rp, rs = _rows(k_rope, ROPE_DIM, T, "k_rope")
    ip, is_ = _rows(index_k, INDEXER_DIM, T, "index_k")
    if bf16_cache:
        mains, idxs, nb = _caches(main_caches, indexer_caches, num_blocks, MAIN_SLOT_BYTES_BF16,
                                  BLOCK_SIZE * INDEXER_SLOT_BYTES_BF16)
    else:
        mains, idxs, nb = _caches(main_caches, indexer_caches, num_blocks)
    cnt = None
    if invalid_count is not None:
        if invalid_count.dtype not in (torch.int64, torch.uint64) or not invalid_count.is_cuda:
            raise ValueError("invalid_count: expected an int64 CUDA tensor")
        cnt = invalid_count.data_ptr()
    tensors = [kv_latent, k_rope, index_k, slot_mapping, *main_caches, *indexer_caches]
    if invalid_count is not None:
        tensors.append(invalid_count)
    check_devices([t.get_device() for t in tensors], _current_device())
    return [lp, ls, rp, rs, ip, is_, slot_mapping.data_ptr(), T, mains, idxs,
            len(main_caches), nb, BLOCK_SIZE, cnt]


def slot_report(slot_mapping, num_blocks: int) -> dict:
    """Debug check of a slot_mapping, on the host (it copies the slots back and
    synchronises, so it is not for the hot path): how many slots are written,
    padded (-1), invalid (other out-of-range values) and duplicated among the
    written ones.  Duplicates leave unspecified bytes in the caches."""
    import numpy as np
    s = slot_mapping.detach().to("cpu").numpy() if isinstance(slot_mapping, torch.Tensor) \
        else np.asarray(slot_mapping)
    s = s.astype(np.int64, copy=False)
    cap = int(num_blocks) * BLOCK_SIZE
    written = s[(s >= 0) & (s < cap)]
    uniq = np.unique(written)
    return {"written": int(written.size), "padded": int(np.count_nonzero(s == -1)),
            "invalid": int(np.count_nonzero((s != -1) & ((s < 0) | (s >= cap)))),
            "duplicates": int(written.size - uniq.size)}


def _check_distinct(slot_mapping, main_caches, num_blocks, main_slot=MAIN_SLOT_BYTES):
    nb = num_blocks if num_blocks is not None else \
        main_caches[0].numel() // (BLOCK_SIZE * main_slot)
    rep = slot_report(slot_mapping, nb)
    if rep["duplicates"]:
        raise ValueError(f"slot_mapping names {rep['duplicates']} slot(s) more than once")


def store_mla_fp8(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                  num_blocks=None, invalid_count=None, stream=None,
                  check_slots: bool = False) -> None:
    """Fused direct publication of every token row into all replicas.
    check_slots=True first runs the host-side slot_report (debug only)."""
    if check_slots:
        _check_distinct(slot_mapping, main_caches, num_blocks)
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count)
    check(lib().kvpub_store_mla_fp8(*args, _stream_handle(stream, _current_device())))


def store_mla_bf16(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                   num_blocks=None, invalid_count=None, stream=None) -> None:
    """Unquantised variant: every row's bf16 bytes into all replicas
    (Main slot 1152 B, Indexer slot 256 B)."""
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count, bf16_cache=True)
    check(lib().kvpub_store_mla_bf16(*args, _stream_handle(stream, _current_device())))


def store_mla_fp8_publish(kv_latent, k_rope, index_k, slot_mapping, main_caches,
                          indexer_caches, epoch, done_count, num_blocks=None,
                          invalid_count=None, stream=None) -> None:
    """Fused publication plus the device-epoch advance, in one launch."""
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count)
    _counter(epoch, (torch.int64, torch.uint64), "epoch")
    _counter(done_count, (torch.int32, torch.uint32), "done_count")
    check(lib().kvpub_store_mla_fp8_publish(*args, epoch.data_ptr(), done_count.data_ptr(),
                                            _stream_handle(stream, _current_device())))


def gather_workspace_bytes(num_tokens: int) -> int:
    return int(lib().kvpub_gather_workspace_bytes(int(num_tokens)))


def gather_insert(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                  workspace, num_blocks=None, invalid_count=None, stream=None) -> None:
    """The unfused path: gather every row, then one insert launch per replica."""
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace: expected a contiguous CUDA tensor")
    check_devices([workspace.get_device()], _current_device())
    nbytes = workspace.numel() * workspace.element_size()
    check(lib().kvpub_gather_insert(*args, workspace.data_ptr(), nbytes,
                                    _stream_handle(stream, _current_device())))


def gather_insert_noalloc(kv_latent, k_rope, index_k, slot_mapping, main_caches,
                          indexer_caches, num_blocks=None, invalid_count=None,
                          stream=None) -> None:
    """gather_insert with the library's fixed workspace, for callers that may
    not allocate device memory (at most STATIC_GATHER_MAX_TOKENS tokens;
    calls that overlap on the GPU race on the shared workspace)."""
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count)
    check(lib().kvpub_gather_insert_noalloc(*args,
                                            _stream_handle(stream, _current_device())))


class PreparedCall:
    """One library call with its arguments marshalled once (shapes checked,
    pointers and the replica pointer arrays built).  Calling it passes only
    the stream, which cuts the per-call host cost of an eager (non-graph)
    serving loop.  The cheapest form passes the raw cudaStream_t handle
    (``torch.cuda.current_stream().cuda_stream``, looked up once per loop):
    with no stream, each call looks up torch's current stream, which costs
    a few microseconds.  It keeps the tensors it was prepared with alive;
    they must not be reallocated while it is in use."""

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, tuple(args), keep
        self._device = _current_device()

    def __call__(self, stream=None) -> None:
        # The default stream is the current device's: if the current device
        # is no longer the one the tensors were checked on, its device index
        # differs and the call is refused (one integer comparison).
        check(self._fn(*self._args, _stream_handle(stream, self._device)))


def prepare_store_mla_fp8(kv_latent, k_rope, index_k, slot_mapping, main_caches,
                          indexer_caches, num_blocks=None, invalid_count=None) -> PreparedCall:
    """store_mla_fp8 with its arguments marshalled once."""
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count)
    keep = (kv_latent, k_rope, index_k, slot_mapping, list(main_caches), list(indexer_caches),
            invalid_count)
    return PreparedCall(lib().kvpub_store_mla_fp8, args, keep)


def prepare_store_mla_fp8_publish(kv_latent, k_rope, index_k, slot_mapping, main_caches,
                                  indexer_caches, epoch, done_count, num_blocks=None,
                                  invalid_count=None) -> PreparedCall:
    """store_mla_fp8_publish with its arguments marshalled once."""
    args = _store_args(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                       num_blocks, invalid_count)
    _counter(epoch, (torch.int64, torch.uint64), "epoch")
    _counter(done_count, (torch.int32, torch.uint32), "done_count")
    keep = (kv_latent, k_rope, index_k, slot_mapping, list(main_caches), list(indexer_caches),
            invalid_count, epoch, done_count)
    return PreparedCall(lib().kvpub_store_mla_fp8_publish,
                        args + [epoch.data_ptr(), done_count.data_ptr()], keep)


def prepare_epoch_advance(epoch) -> PreparedCall:
    """epoch_advance with its argument marshalled once."""
    _counter(epoch, (torch.int64, torch.uint64), "epoch")
    return PreparedCall(lib().kvpub_epoch_advance, [epoch.data_ptr()], (epoch,))


def _counter(t, dtypes, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in dtypes or t.numel() < 1:
        raise ValueError(f"{name}: expected a CUDA tensor of {dtypes}")
    check_devices([t.get_device()], _current_device())


def epoch_advance(epoch: torch.Tensor, stream=None) -> None:
    """Release all earlier stores on the stream, then add 1 to ``epoch``."""
    _counter(epoch, (torch.int64, torch.uint64), "epoch")
    check(lib().kvpub_epoch_advance(epoch.data_ptr(),
                                    _stream_handle(stream, _current_device())))


def epoch_wait(epoch: torch.Tensor, target: int, max_polls: int, status: torch.Tensor,
               stream=None) -> None:
    """Bounded acquire-wait until ``epoch >= target``; writes 0 (ok) / 1 (timeout)."""
    _counter(epoch, (torch.int64, torch.uint64), "epoch")
    _counter(status, (torch.int32, torch.uint32), "status")
    check(lib().kvpub_epoch_wait(epoch.data_ptr(), int(target), int(max_polls),
                                 status.data_ptr(), _stream_handle(stream, _current_device())))
