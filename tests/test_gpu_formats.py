"""GPU parity of the MXFP4 helpers and the device input generator (bit-exact)."""
import numpy as np
import pytest
import torch

from bit_expert_ffn_moe_gb300 import binding as B
from bit_expert_ffn_moe_gb300 import inputs as IN
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host_generator():
    rows, K = 96, 640
    c = IN.weight_scale(0.02)
    out = torch.empty((3, rows, K), dtype=torch.float32, device="cuda")
    B.moe_synth_weights(1234, 2, 5, 3, rows, K, float(c), out)
    got = out.cpu().numpy()
    for n in range(3):
        ref = IN.synth_weights(1234, 2, 5 + n, rows, K, 0.02)
        np.testing.assert_array_equal(got[n], ref)


def _adversarial_rows():
    rng = np.random.default_rng(21)
    rows = [rng.standard_normal(256) * 0.02,
            rng.standard_normal(256) * np.exp(rng.uniform(-60, 60)),
            np.zeros(256), -np.zeros(256)]
    # every tie point and grid value, scaled into blocks with amax 6 * 2^X
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1, 1.5, 2, 3, 4, 0, 5.9] * 2)
    for X in (-20, 0, 7):
        v = ties * 2.0 ** X
        v[::3] *= -1
        rows.append(np.concatenate([v] * 8))
    tiny = np.full(256, 1e-40)
    tiny[0] = 1e-38
    rows.append(tiny)
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("kind", ["synth", "adversarial"])
def test_pack_and_unpack_match_oracle(kind):
    if kind == "synth":
        w = IN.synth_weights(99, 0, 0, 512, 1024, 0.02)
    else:
        w = _adversarial_rows()
    rows, K = w.shape
    wd = torch.from_numpy(w).cuda()
    q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    B.moe_mxfp4_pack(wd, rows, K, q, s)
    q_ref, s_ref = O.mxfp4_pack(w)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    back = torch.empty_like(wd)
    B.moe_mxfp4_unpack(q, s, rows, K, back)
    np.testing.assert_array_equal(back.cpu().numpy(), O.mxfp4_unpack(q_ref, s_ref))


def test_scales_to_mma_layout():
    rows, K = 384, 512
    s = np.random.default_rng(3).integers(0, 255, size=(rows, K // 32)).astype(np.uint8)
    out = torch.empty(B.moe_mxfp4_mma_scale_bytes(rows, K), dtype=torch.uint8, device="cuda")
    B.moe_mxfp4_scales_to_mma(torch.from_numpy(s).cuda(), rows, K, out)
    got = out.cpu().numpy()
    # documented layout: atom (R, C) at index R*(K/128) + C; row r, column c inside it at
    # (r%32)*16 + ((r/32)%4)*4 + c%4
    ref = np.empty_like(got)
    for r in range(rows):
        for c in range(K // 32):
            atom = (r // 128) * (K // 128) + c // 4
            ref[atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4] = s[r, c]
    np.testing.assert_array_equal(got, ref)


def _tiles_reference(virt_codes, K):
    """Documented code tiles of a [rows][K/2] code matrix: tile (R, C) at index R*(K/256) + C,
    16-byte chunk j of row r inside it at r*128 + (j ^ (r % 8))*16."""
    rows = virt_codes.shape[0]
    out = np.empty(rows * K // 2, dtype=np.uint8)
    for r in range(rows):
        for b in range(K // 32):
            tile = (r // 128) * (K // 256) + b // 8
            off = tile * 16384 + (r % 128) * 128 + ((b % 8) ^ (r % 8)) * 16
            out[off:off + 16] = virt_codes[r, 16 * b:16 * b + 16]
    return out


def test_codes_to_mma_tiles():
    rows, K = 256, 512
    q = np.random.default_rng(5).integers(0, 256, size=(rows, K // 2)).astype(np.uint8)
    out = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    B.moe_mxfp4_codes_to_mma(torch.from_numpy(q).cuda(), rows, K, out)
    np.testing.assert_array_equal(out.cpu().numpy(), _tiles_reference(q, K))
