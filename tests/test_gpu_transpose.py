"""GPU parity of the tiled transpose (tgemm_transpose) against the oracle
(oracle/transpose.py): bit-exact, for 2- and 4-byte elements, ragged edges,
row padding on both sides, 16-byte and unaligned rows, and guard bands that
must stay untouched."""
import numpy as np
import pytest
import torch

from oracle import transpose as ot
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

CANARY = {2: 0x7E5A, 4: 0x7FA1B2C3}
BITS = {2: np.uint16, 4: np.uint32}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    H.tg()
    torch.cuda.set_device(0)


def run(rows, cols, eb, ld_src=None, ld_dst=None, src_off=0, dst_off=0, seed=0):
    lib = H.tg()
    dev = torch.device("cuda:0")
    ld_src = cols if ld_src is None else ld_src
    ld_dst = rows if ld_dst is None else ld_dst
    rng = np.random.default_rng(seed)
    src = rng.integers(0, 2 ** (8 * eb) - 1, size=(rows, ld_src), dtype=np.uint64).astype(BITS[eb])
    guard = 64
    dst_init = np.full(guard + cols * ld_dst + guard, CANARY[eb], dtype=BITS[eb])
    s_buf, s_ptr = H.upload(src, src_off, dev)
    d_buf, d_base = H.upload(dst_init, dst_off, dev)
    d_ptr = d_base + guard * eb
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib.transpose(rows, cols, s_ptr, ld_src, d_ptr, ld_dst, eb, stream)
    assert st == lib.OK, lib.status_string(st)
    assert lib.device_status(stream) == lib.OK
    start = d_base - d_buf.data_ptr()
    raw = d_buf[start:start + dst_init.size * eb].cpu().numpy().view(BITS[eb])
    assert np.all(raw[:guard] == CANARY[eb]) and np.all(raw[guard + cols * ld_dst:] == CANARY[eb]), "guard band"
    body = raw[guard:guard + cols * ld_dst].reshape(cols, ld_dst)
    want = ot.transpose(src, rows, cols, np.full((cols, ld_dst), CANARY[eb], dtype=BITS[eb]), ld_dst)
    assert np.array_equal(body, want), "transpose differs from the oracle (or padding written)"


@pytest.mark.parametrize("eb", [2, 4])
@pytest.mark.parametrize("shape", [(1, 1), (7, 9), (64, 64), (65, 63), (128, 192), (300, 520), (1000, 1500)],
                         ids=lambda s: "x".join(map(str, s)))
def test_transpose_shapes(shape, eb):
    rows, cols = shape
    run(rows, cols, eb, seed=rows * 7 + cols)


@pytest.mark.parametrize("eb", [2, 4])
@pytest.mark.parametrize("lds,offs", [((520, 300), (0, 0)), ((528, 304), (0, 0)), ((530, 301), (0, 0)),
                                      ((520, 300), (4, 2)), ((536, 312), (16, 32))],
                         ids=["dense", "padded16", "padded_odd", "misaligned_base", "aligned_offsets"])
def test_transpose_pitches_and_alignment(lds, offs, eb):
    rows, cols = 300, 520
    if offs[0] % eb or offs[1] % eb:
        pytest.skip("offset not a multiple of the element size")
    run(rows, cols, eb, ld_src=lds[0], ld_dst=lds[1], src_off=offs[0], dst_off=offs[1], seed=3)


def test_transpose_large_f32():
    run(4096, 6144, 4, seed=11)
