"""The read-then-pin pool reader on the CPU ([Review] §2.7, fast engine start).

ft_pool_read fills host memory from a pool file with several threads.  These
tests need no GPU: they read into ordinary (and freshly mapped) host memory
and compare bytes, including offsets, odd sizes, more threads than pieces, a
file that ends early and a file that does not exist.
"""
import os

import numpy as np
import pytest


@pytest.fixture(scope="module")
def pool_file(tmp_path_factory):
    d = np.random.default_rng(11).integers(0, 256, size=(3 << 20) + 12345, dtype=np.uint8)
    path = str(tmp_path_factory.mktemp("pool") / "pool.bin")
    d.tofile(path)
    return path, d


@pytest.mark.parametrize("offset,nbytes,threads", [
    (0, (3 << 20) + 12345, 1),
    (0, (3 << 20) + 12345, 7),
    (4096, 1 << 20, 0),
    (777, 1000, 64),
    (5, 3, 4),
])
def test_pool_read_copies_the_file_range(ftlib, pool_file, offset, nbytes, threads):
    path, d = pool_file
    dst = np.full(nbytes + 64, 0xA5, dtype=np.uint8)
    ftlib.ft_pool_read(path, offset, dst.ctypes.data, nbytes, threads)
    assert np.array_equal(dst[:nbytes], d[offset:offset + nbytes])
    assert (dst[nbytes:] == 0xA5).all()          # nothing written past the range


def test_pool_read_into_a_fresh_mapping(ftlib, pool_file):
    path, d = pool_file
    buf = ftlib.RegisteredBuffer(d.size)
    buf.read(path, 0, 5)
    assert np.array_equal(buf.tensor.numpy(), d)
    assert buf.ptr % 4096 == 0
    buf.free()


def test_pool_read_errors(ftlib, pool_file, tmp_path):
    path, d = pool_file
    dst = np.zeros(d.size + 100, dtype=np.uint8)     # room for more than the file holds
    with pytest.raises(ftlib.FTError) as ei:
        ftlib.ft_pool_read(path, 0, dst.ctypes.data, d.size + 100, 3)
    assert ei.value.status == ftlib.FT_EIO
    with pytest.raises(ftlib.FTError) as ei:
        ftlib.ft_pool_read(str(tmp_path / "missing.bin"), 0, dst.ctypes.data, 10, 1)
    assert ei.value.status == ftlib.FT_EIO
    with pytest.raises(ftlib.FTError) as ei:
        ftlib.ft_pool_read(path, 0, dst.ctypes.data, 10, 257)
    assert ei.value.status == ftlib.FT_EINVAL
    ftlib.ft_pool_read(path, 0, 0, 0, 1)               # an empty read is a no-op
    assert os.path.getsize(path) == d.size


def test_injection_sites_validate(ftlib):
    with pytest.raises(ftlib.FTError):
        ftlib.ft_debug_inject_failure(0, 1)
    with pytest.raises(ftlib.FTError):
        ftlib.ft_debug_inject_failure(4, 1)
    for site in (ftlib.FT_INJECT_DEVICE_ALLOC, ftlib.FT_INJECT_HOST_PIN, ftlib.FT_INJECT_STREAM_EVENT):
        ftlib.ft_debug_inject_failure(site, -1)
    assert ftlib.ft_debug_live_resources() == (0, 0)
