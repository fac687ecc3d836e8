"""moe_sort_by_expert_noalloc: the expert sort on the library's fixed device scratch.

Compared bit-exactly with moe_sort_by_expert (caller workspace) and with the oracle's stable
counting sort on two calls issued back to back on one stream, which reuse the same scratch;
the file is named to be collected last so it also runs after every other GPU test in the
session.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

KEYS = ("sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm")


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


def _ids_glm(T=2048, E=160, k=8):
    case = S.workload("c2")
    ids, _ = O.route_topk(case.logits[:T], k)
    return torch.from_numpy(ids).cuda(), E


def _ids_ragged():
    # 37 tokens, 3 slots, 5 experts, with unfilled (-1) slots
    g = np.random.default_rng(7)
    ids = np.stack([g.permutation(5)[:3] for _ in range(37)]).astype(np.int32)
    ids[g.random(ids.shape) < 0.1] = -1
    return torch.from_numpy(ids).cuda(), 5


def _alloc(ids, E):
    T, k = ids.shape
    d = ids.device
    return dict(sorted_token_ids=torch.full((T * k,), -7, dtype=torch.int32, device=d),
                sorted_expert_ids=torch.full((T * k,), -7, dtype=torch.int32, device=d),
                expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=d),
                token_to_perm=torch.full((T, k), -7, dtype=torch.int32, device=d))


def test_two_calls_in_a_row_match_the_workspace_sort():
    cases = [_ids_glm(), _ids_ragged()]
    outs = [_alloc(ids, E) for ids, E in cases]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for (ids, E), out in zip(cases, outs):  # back to back, same scratch, no sync between
            moe.moe_sort_by_expert_noalloc(ids, E, out=out, stream=s)
    s.synchronize()
    for (ids, E), out in zip(cases, outs):
        ref = moe.moe_sort_by_expert(ids, E)
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(out[key], ref[key]), key
        # and directly against the oracle's stable counting sort, bit for bit
        srt = O.sort_by_expert(ids.cpu().numpy(), E)
        for key in KEYS:
            np.testing.assert_array_equal(out[key].cpu().numpy().reshape(srt[key].shape), srt[key], err_msg=key)


def test_repeated_call_is_identical():
    ids, E = _ids_glm(T=333, k=8)
    a = moe.moe_sort_by_expert_noalloc(ids, E)
    b = moe.moe_sort_by_expert_noalloc(ids, E)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(a[key], b[key]), key


def test_problem_above_the_scratch_limit_is_refused():
    ids = torch.zeros(104200, 8, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_sort_by_expert_noalloc(ids, 160)
    assert "MOE_ERR_SCRATCH_LIMIT" in str(ei.value)
