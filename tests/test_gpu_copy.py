"""GPU: qlora_copy_many, the host <-> device copy call the end-to-end step uses.

Byte-exact round trips through pinned host memory and device memory for sizes
below, at and above the 2 MB piece size (odd byte counts included), several
copies in one call, the empty list, a NULL pointer, and the call inside a CUDA
graph capture (fork to the copy streams and join back as graph edges).
"""

import pytest
import torch

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 17, 4096, (2 << 20) + 5, 16 * (1 << 20) + 3]


def _host_bytes(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory()


def test_round_trip_bytes_exact(lib):
    hosts = [_host_bytes(n, i) for i, n in enumerate(SIZES)]
    devs = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in SIZES]
    lib.copy_many(list(zip(devs, hosts)))
    devs2 = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in SIZES]
    lib.copy_many(list(zip(devs2, devs)))  # device to device
    backs = [torch.zeros(n, dtype=torch.uint8).pin_memory() for n in SIZES]
    lib.copy_many(list(zip(backs, devs2)))
    torch.cuda.synchronize()
    lib.check_status()
    for h, b in zip(hosts, backs):
        assert torch.equal(h, b)


def test_stream_order_with_kernels(lib):
    """The copies are ordered after earlier work and before later work of the caller's stream."""
    n = 8 << 20
    h = _host_bytes(n, 7)
    d = torch.zeros(n, dtype=torch.uint8, device="cuda")
    d.add_(1)  # earlier work on the stream writes d ...
    lib.copy_many([(d, h)])  # ... and the copy overwrites it afterwards
    d2 = d.clone()  # later work reads the copied bytes
    torch.cuda.synchronize()
    assert torch.equal(d2.cpu(), h)


def test_empty_list_and_null_pointer(lib):
    lib.copy_many([])
    err = lib.load().qlora_copy_many(None, 1, None)
    assert err == lib.QLORA_ERR_INVALID_ARGUMENT


def test_inside_graph_capture(lib):
    n = (3 << 20) + 11
    h = _host_bytes(n, 9)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        lib.copy_many([(d, h)])
        out.copy_(d)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), h)
