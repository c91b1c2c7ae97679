"""dbf_pack / dbf_unpack on the GPU against the oracle's packing (bit-exact)."""

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,ldw", [(1, 1, 1), (3, 31, 1), (5, 32, 1), (7, 33, 2), (16, 257, 12),
                                           (64, 4096, 128), (100, 5013, 157), (37, 5013, 160), (4096, 32, 1)])
def test_pack_matches_oracle_bit_exact(cuda_lib, rows, cols, ldw):
    rng = np.random.default_rng(rows * 7919 + cols)
    s = np.where(rng.random((rows, cols)) < 0.5, 1, -1).astype(np.int8)
    words = cuda_lib.pack(torch.from_numpy(s).cuda(), ldw)
    torch.cuda.synchronize()
    got = words.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, O.pack_signs(s, ldw))
    back = cuda_lib.unpack(words, cols).cpu().numpy()
    assert np.array_equal(back, s)


def test_pack_maps_only_positive_to_one(cuda_lib):
    rng = np.random.default_rng(5)
    s = rng.integers(-128, 128, size=(9, 70)).astype(np.int8)
    s[0, :5] = 0
    words = cuda_lib.pack(torch.from_numpy(s).cuda(), 3)
    assert np.array_equal(words.cpu().numpy().view(np.uint32), O.pack_signs(s, 3))


def test_pack_golden_fixtures(cuda_lib, golden_dir):
    import json, os
    with open(os.path.join(golden_dir, "pack_format.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        s = np.asarray([[1 if ch == "+" else -1 for ch in c["signs"]]], dtype=np.int8)
        words = cuda_lib.pack(torch.from_numpy(s).cuda(), c["ldw"]).cpu().numpy().view(np.uint32)
        assert [int(w) for w in words[0]] == [int(w, 16) for w in c["words"]], c["name"]
