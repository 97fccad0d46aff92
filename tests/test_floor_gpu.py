"""The measurement reference kernels (frn_floor_launch): the copy kernel
stores the xor of its sources' vectors into both outputs, over a ragged last
CTA; the read and empty kernels run; bad arguments launch nothing."""
import pytest
import torch

import reduce_residual_rmsnorm_fp32_gb300 as frn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_src,nbytes,threads", [(9, 7168 * 2 * 8, 128), (1, 16, 32), (17, 4096 * 2 * 37 + 48, 256)])
def test_floor_copy_stores_the_xor(n_src, nbytes, threads):
    g = torch.Generator(device="cuda")
    g.manual_seed(n_src)
    srcs = [torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), generator=g, device="cuda", dtype=torch.int32)
            for _ in range(n_src)]
    d0 = torch.full((nbytes // 4,), 7, device="cuda", dtype=torch.int32)
    d1 = torch.full_like(d0, 9)
    frn.floor_launch(frn.FLOOR_COPY, srcs, d0, d1, threads=threads)
    frn.floor_launch(frn.FLOOR_READ, srcs, threads=threads)
    frn.floor_launch(frn.FLOOR_EMPTY, threads=threads, grid=3)
    torch.cuda.synchronize()
    want = srcs[0].clone()
    for t in srcs[1:]:
        want ^= t
    assert torch.equal(d0, want) and torch.equal(d1, want)


def test_floor_rejects_bad_arguments():
    a = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(frn.FrnError):
        frn.floor_launch(3, [a])
    with pytest.raises(frn.FrnError):
        frn.floor_launch(frn.FLOOR_COPY, [a], a, None)
    with pytest.raises(frn.FrnError):
        frn.floor_launch(frn.FLOOR_READ, [a], threads=48)
    with pytest.raises(ValueError):
        frn.floor_launch(frn.FLOOR_COPY, [a], a[:8], a)
