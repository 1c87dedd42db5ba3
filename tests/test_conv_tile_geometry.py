"""The stride-2 conv kernels' work decoding (csrc/ito_conv_tc.cu), restated on the host:
for the parity-phase delta propagation every element of the input-space delta is written
by exactly one 32 x 32 store box, with in-range box origins and 16-byte aligned x; the
forward's row tiles are runs of 128 consecutive output positions and the weight
gradient's position blocks runs of 64; and each tap reads the parity plane and shift of
y = 2 oh + kh - 1. Shapes: the CNN's second and third convs at batch 128 and the
parity-plane cases of the GPU tests."""
import pytest

SHAPES = [(128, 32, 32, 64, 128), (128, 16, 16, 128, 256), (1, 16, 16, 64, 64), (3, 16, 16, 128, 64),
          (2, 64, 64, 64, 64), (2, 4, 32, 64, 128), (2, 16, 16, 64, 512)]


def eligible(B, H, W, IC, OC):
    OH, OW = H // 2, W // 2
    pow2 = OH > 0 and OH & (OH - 1) == 0
    return H % 2 == 0 and W % 2 == 0 and OW in (8, 16, 32) and pow2 and OH * OW >= 32 and IC % 64 == 0 \
        and OC % 64 == 0


def phase_of(po):
    # the phases in the order their tiles are handed out: (1,1), (1,0), (0,1), (0,0)
    return (0 if po in (2, 3) else 1), (0 if po in (1, 3) else 1)


@pytest.mark.parametrize("B,H,W,IC,OC", SHAPES)
def test_phase_kernel_writes_every_delta_element_once(B, H, W, IC, OC):
    assert eligible(B, H, W, IC, OC)
    OH, OW = H // 2, W // 2
    bn = 128 if IC % 128 == 0 else 64
    oha = min(OH, 128 // OW)
    ba = 128 // (OW * oha)
    n_iblk = OH // oha
    m_tiles = -(-B // ba) * n_iblk
    n_tiles = IC // bn
    per = m_tiles * n_tiles
    written = {}
    for w in range(4 * per):
        po, r = divmod(w, per)
        mt, nt = divmod(r, n_tiles)
        py, px = phase_of(po)
        b0, i0 = (mt // n_iblk) * ba, (mt % n_iblk) * oha
        for quad in range(4):
            r0 = quad * 32
            b_off, rem = divmod(r0, oha * OW)
            i_off, j_off = divmod(rem, OW)
            assert j_off == 0 and i_off + 32 // OW <= oha
            b = b0 + b_off
            if b >= B:
                continue
            for half in range(2):
                for gq in range(bn // 64):
                    x = nt * bn + half * (bn // 2) + gq * 32
                    assert (x * 4) % 16 == 0
                    for ii in range(32 // OW):
                        i = i0 + i_off + ii
                        assert 0 <= i < OH
                        key0 = (b, 2 * i + py)
                        for j in range(OW):
                            k = key0 + (2 * j + px, x)
                            written[k] = written.get(k, 0) + 1
    # each key stands for a 32-channel run; every run exactly once
    assert len(written) == B * H * W * (IC // 32)
    assert set(written.values()) == {1}


@pytest.mark.parametrize("B,H,W,IC,OC", SHAPES)
def test_plane_kernel_tiles_are_consecutive_positions(B, H, W, IC, OC):
    OH, OW = H // 2, W // 2
    oha = min(OH, 128 // OW)
    ba = 128 // (OW * oha)
    n_iblk = OH // oha
    for mt in range(-(-B // ba) * n_iblk):
        b0, i0 = (mt // n_iblk) * ba, (mt % n_iblk) * oha
        flat = [((b0 + bl) * OH + i0 + il) * OW + j for bl in range(ba) for il in range(oha) for j in range(OW)]
        r0 = (b0 * OH + i0) * OW
        assert flat == list(range(r0, r0 + 128))
    ohb = min(OH, 64 // OW)
    bb = 64 // (OW * ohb)
    n_iblk_w = OH // ohb
    for kb in range(-(-B // bb) * n_iblk_w):
        b0, i0 = (kb // n_iblk_w) * bb, (kb % n_iblk_w) * ohb
        flat = [((b0 + bl) * OH + i0 + il) * OW + j for bl in range(bb) for il in range(ohb) for j in range(OW)]
        assert flat == list(range(64 * kb, 64 * kb + 64))


def test_taps_read_the_right_plane_and_shift():
    for kh in range(3):
        py, sh = (kh + 1) & 1, (-1 if kh == 0 else 0)
        for oh in range(16):
            assert 2 * (oh + sh) + py == 2 * oh + kh - 1
    # delta phases: input row 2i + py receives kernel row kh from output row i + dh
    for py, taps in ((0, [(0, 1)]), (1, [(1, 0), (0, 2)])):
        for i in range(8):
            y = 2 * i + py
            got = sorted((i + dh, kh) for dh, kh in taps)
            want = sorted((oh, kh) for kh in range(3) for oh in range(10) if 2 * oh + kh - 1 == y)
            assert got == want
