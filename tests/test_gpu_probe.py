"""The streaming-read probe (the host-link roofline's denominator): every
16-byte chunk of the buffer is read exactly once, whatever the launch shape,
from device memory and from pinned host memory read in place.

Check: each block writes the XOR of its threads' folds of the chunks they
read, (x ^ z) << 32 | (y ^ w) per chunk of words (x, y, z, w); XOR is
associative and commutative, so the XOR of all sink words equals the XOR of
that fold over every chunk of the buffer, computed here with numpy."""
import numpy as np
import pytest
import torch

from offloaded_kv_cache_gb300 import kvsparse as kv

pytestmark = pytest.mark.gpu


def expected_fold(buf: np.ndarray) -> int:
    w = buf.view(np.uint32).reshape(-1, 4).astype(np.uint64)
    fold = ((w[:, 0] ^ w[:, 2]) << np.uint64(32)) | (w[:, 1] ^ w[:, 3])
    return int(np.bitwise_xor.reduce(fold))


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("blocks,threads,loads", [(1, 128, 4), (7, 256, 8), (300, 512, 16),
                                                  (152, 1024, 4)])
def test_probe_reads_every_chunk_once(kvlib, where, blocks, threads, loads):
    rng = np.random.default_rng(blocks + threads + loads)
    nbytes = (3 << 20) + 16 * 37                 # not a multiple of the grid's stride
    data = rng.integers(0, 256, nbytes, dtype=np.uint8)
    src = torch.from_numpy(data)
    src = src.pin_memory() if where == "host" else src.cuda()
    sink = torch.zeros(blocks, dtype=torch.int64, device="cuda")
    kv.kv_stream_read_probe_shape(src, nbytes, sink, blocks, threads, loads)
    torch.cuda.synchronize()
    got = int(np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint64)))
    assert got == expected_fold(data)


def test_probe_default_shape_and_refusals(kvlib):
    data = np.arange(1 << 20, dtype=np.uint32).view(np.uint8)
    src = torch.from_numpy(data).cuda()
    sink = torch.zeros(4096, dtype=torch.int64, device="cuda")
    kv.kv_stream_read_probe(src, data.size, sink)
    torch.cuda.synchronize()
    assert int(np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint64))) == expected_fold(data)
    for blocks, threads, loads in [(0, 256, 4), (4, 96, 4), (4, 256, 5), (4, 2048, 4)]:
        rc = kv.kv_stream_read_probe_shape(src, data.size, sink, blocks, threads, loads,
                                           check=False)
        assert rc == kv.KV_ERR_INVALID_ARG
    rc = kv.kv_stream_read_probe_shape(src, 24, sink, 4, 256, 4, check=False)   # not 16 x n
    assert rc == kv.KV_ERR_INVALID_ARG
