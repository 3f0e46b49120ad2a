"""GPU: the load-time import of GGUF-style Q4 blocks through the C ABI
(moe_import_q4_blocks) against the oracle, bit for bit: the decoded fp32
weights, the packed int4 bytes and the fp16 scales, at groups inside one block
(8, 16, 32: the block kept exactly) and across blocks (64, 128: re-quantised).  The block layout and the
import follow the oracle's reading R15 (the Q4 weight load from GGUF of
thewafflehaus/butter PR #69, commit "feat(laguna): Laguna-S-2.1 decode on the
CUDA engine")."""
import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import oracle

pytestmark = pytest.mark.gpu


def random_blocks(rng, rows, K):
    """Every code byte uniform; scales finite fp16 of both signs over the normal range,
    one block with scale 0."""
    nb = K // 32
    blocks = rng.integers(0, 256, size=(rows, nb, 18), dtype=np.uint8)
    mag = np.exp2(rng.integers(-14, 8, size=(rows, nb))) * (1 + rng.integers(0, 1024, (rows, nb)) / 1024)
    d = (mag * rng.choice([-1.0, 1.0], size=(rows, nb))).astype(np.float16)
    d[0, 0] = 0.0
    bits = d.view(np.uint16)
    blocks[:, :, 0] = (bits & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (bits >> 8).astype(np.uint8)
    return blocks.reshape(rows, nb * 18)


@pytest.mark.parametrize("rows,K,g", [(1, 32, 32), (3, 96, 32), (2, 64, 8), (4, 160, 16),
                                      (5, 256, 128), (7, 384, 64), (33, 4096, 128)])
def test_import_matches_oracle(rows, K, g):
    rng = np.random.default_rng(rows * 1000 + K + g)
    blocks = random_blocks(rng, rows, K)
    q, s, w = moe.moe_import_q4_blocks(torch.from_numpy(blocks).cuda(), K, g)
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy(), oracle.dequant_q4_blocks(blocks, K))
    qo, so = oracle.import_q4_blocks(blocks, K, g)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), so)


@pytest.mark.parametrize("sfx,nbytes", [("", 18), ("64", 36)])
def test_import_hand_worked_fixture_on_gpu(sfx, nbytes):
    """Case A (group 32: the block kept exactly) and case B (group 64 across two
    blocks: re-quantised)."""
    from conftest import read_golden
    gold = read_golden("q4_block_example.txt")
    K, g = int(gold["K" + sfx][0][0]), int(gold["group" + sfx][0][0])
    block = np.array([int(v, 16) for v in gold["block" + sfx][0]], np.uint8).reshape(1, nbytes)
    q, s, _ = moe.moe_import_q4_blocks(torch.from_numpy(block).cuda(), K, g)
    torch.cuda.synchronize()
    assert q.cpu().numpy().tobytes().hex().upper() == "".join(gold["bytes" + sfx][0])
    assert [f"{v:04X}" for v in s.cpu().numpy().view(np.uint16)[0]] == gold["scales" + sfx][0]
