"""mla_copy_from_host: a kernel that reads page-locked host memory over the bus.

Byte-exact copies for aligned and unaligned sizes and offsets, and the argument checks
(pageable host memory and device memory as the source are refused before any launch).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import head_latent_attention_25_b300 as pkg
    return pkg


@pytest.mark.parametrize("nbytes,src_off,dst_off", [
    (1, 0, 0), (15, 0, 0), (16, 0, 0), (4096 + 3, 0, 0), (1 << 20, 0, 0),
    (4 * 1024 * 1024 + 16 * 7, 0, 0), (1000, 1, 0), (1000, 0, 3), (65536, 8, 8)])
def test_copy_bytes_exact(nbytes, src_off, dst_off):
    pkg = _lib()
    g = torch.Generator().manual_seed(nbytes)
    host = torch.randint(0, 256, (nbytes + 32,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes + 32,), 0xAB, dtype=torch.uint8, device="cuda")
    pkg.mla_copy_from_host(dev.data_ptr() + dst_off, host.data_ptr() + src_off, nbytes,
                           torch.cuda.current_stream())
    torch.cuda.synchronize()
    got = dev.cpu()
    assert torch.equal(got[dst_off:dst_off + nbytes], host[src_off:src_off + nbytes])
    # nothing outside the destination range was touched
    assert bool((got[:dst_off] == 0xAB).all()) and bool((got[dst_off + nbytes:] == 0xAB).all())


def test_copy_zero_bytes_is_a_no_op():
    pkg = _lib()
    n0 = pkg.mla_launch_count()
    pkg.mla_copy_from_host(0, 0, 0)
    assert pkg.mla_launch_count() == n0


def test_copy_refuses_pageable_and_device_sources():
    pkg = _lib()
    dev = torch.empty(4096, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(4096, dtype=torch.uint8)
    other = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    for src in (pageable, other):
        with pytest.raises(pkg.MlaError) as e:
            pkg.mla_copy_from_host(dev, src, 4096)
        assert e.value.status == pkg.MLA_ERR_INVALID_ARG
    pinned = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    with pytest.raises(pkg.MlaError) as e:            # destination in host memory
        pkg.mla_copy_from_host(pinned, pinned, 4096)
    assert e.value.status == pkg.MLA_ERR_INVALID_ARG
