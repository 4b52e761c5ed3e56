"""Request life cycles on one cache: requests are released and refilled (their pages recycled
through the free list, their recorded value-scale maxima reset) while the others keep decoding,
with chunked prefill of new prompts, fused decode steps and multi-request appends interleaved.

Each request mirrors its tokens in an oracle cache, which is reset when the request is released.
After every operation the attention of each request (fused decode steps, and chunked-prefill
queries) is checked against the oracle, and at the end every stored INT2 and BF16 byte.  A refill
uses values 1000 times smaller than the request's previous life, so a maximum that was not reset
would shrink its probabilities' range and show up in the comparison.  Bars: rel-L2 <= 1e-3,
max-abs <= 2e-3 (relative to the largest output).
Sources: axbrief.com OSCAR page, sections "attention-statistics rotation + Triton kernels" and
"OSCAR release" (write and read paths, paged cache with BF16 sink and window).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K
from gpu_util import check_bf16_bytes, check_int2_bytes, oracle_rk, pages_needed, rel_l2

pytestmark = pytest.mark.gpu

B, HQ, HKV = 3, 16, 2
G = HQ // HKV
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_rotated_paged_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    K.oscar_set_decode_path(K.PATH_WARP_MMA)


def _bits_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def test_release_refill_decode_and_prefill_cycles():
    rk = oracle_rk(77, HKV, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    per_seq = pages_needed(2400) + 2
    cache = K.Cache(B, HQ, HKV, per_seq * B + 4, per_seq, page_order=synth.page_order(5, per_seq * B + 4, "permuted"))
    rng = np.random.default_rng(123)
    life = [0] * B            # how often each request was refilled
    ocs = {}                  # (b, h) -> oracle cache of the request's current life

    def fresh(b):
        for h in range(HKV):
            ocs[(b, h)] = oracle.OracleCache(rk[h])

    for b in range(B):
        fresh(b)

    def tokens(b, n):
        scale = 1000.0 ** (-life[b])
        k = rng.standard_normal((n, HKV, D)).astype(np.float32)
        v = (rng.standard_normal((n, HKV, D)) * scale).astype(np.float32)
        kb = synth.bf16_bits(torch.tensor(k).to(torch.bfloat16))
        vb = synth.bf16_bits(torch.tensor(v).to(torch.bfloat16))
        return kb, vb

    def append(n):
        ks, vs = [], []
        for b in range(B):
            kb, vb = tokens(b, n[b])
            ks.append(kb)
            vs.append(vb)
            for h in range(HKV):
                if n[b]:
                    ocs[(b, h)].append(kb[:, h], vb[:, h])
        k = _bits_tensor(np.concatenate(ks)).cuda()
        v = _bits_tensor(np.concatenate(vs)).cuda()
        return k, v

    def check(out, q, qrows, last=None):
        got = out.float().cpu().numpy()
        qh = q.float().cpu().numpy()
        for (b, r) in qrows:
            for h in range(HKV):
                oc = ocs[(b, h)]
                if last is None:
                    ref, _ = oc.attend(qh[r, h * G:(h + 1) * G])
                else:
                    ref, _ = oc.attend_upto(qh[r, h * G:(h + 1) * G], last[(b, r)])
                o = got[r, h * G:(h + 1) * G]
                scale = max(1e-30, float(np.abs(ref).max()))
                assert rel_l2(o, ref) <= 1e-3 and float(np.abs(o - ref).max()) <= 2e-3 * scale, (b, r, h, life[b])

    def decode_steps(n_steps):
        out = torch.empty(B, HQ, D, device="cuda")
        for _ in range(n_steps):
            if min(cache.length(b) for b in range(B)) == 0:
                return
            k, v = append([1] * B)
            q = torch.tensor(rng.standard_normal((B, HQ, D)).astype(np.float32), device="cuda")
            cache.step(k, v, q, rk_dev, out)
            torch.cuda.synchronize()
            check(out, q, [(b, b) for b in range(B)])

    def prefill(n, n_attend=48):
        # append a prompt of n[b] tokens per request, then chunked-prefill attention for its last
        # min(n[b], n_attend) tokens (each query sees the positions up to its own)
        k, v = append(n)
        cache.append(k, v, n, rk_dev)
        nq = [min(x, n_attend) for x in n]
        lens1 = [cache.length(b) for b in range(B)]
        q = torch.tensor(rng.standard_normal((max(1, sum(nq)), HQ, D)).astype(np.float32), device="cuda")
        out = torch.empty_like(q)
        ws = cache.prefill(q, nq, rk_dev, out)
        K.oscar_decode_status(cache.handle, ws)    # no bounded wait gave up
        torch.cuda.synchronize()
        rows, last, r = [], {}, 0
        for b in range(B):
            for i in range(nq[b]):
                rows.append((b, r))
                last[(b, r)] = lens1[b] - nq[b] + i
                r += 1
        check(out, q, rows, last)

    prefill([900, 400, 1200])
    decode_steps(5)
    for cycle in range(3):
        b = cycle % B
        K.kv_page_table_release(cache.handle, b)
        life[b] += 1
        fresh(b)
        n = [0] * B
        n[b] = int(rng.integers(300, 1500))
        prefill(n)                     # the refilled request's prompt, the others idle
        decode_steps(4)
        n = [int(x) for x in rng.integers(0, 200, B)]
        prefill(n)                     # more prompt text for everyone
        decode_steps(3)
    torch.cuda.synchronize()
    for (b, h), oc in ocs.items():
        check_int2_bytes(cache, oc, b, h)
        check_bf16_bytes(cache, oc, b, h)
    assert all(cache.length(b) == ocs[(b, 0)].length for b in range(B))
