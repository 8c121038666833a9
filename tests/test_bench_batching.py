"""bench.py's continuous-batching measurement, run on the CPU against a
stand-in for the library's batcher: the accounting of steps, token steps and
generated tokens, and the page sizing.  The stand-in follows the scheduler's
documented rules: a sequence with a p-token prompt and n new tokens holds its
slot for p + n - 1 steps, and waiting sequences are admitted as slots free."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _FakeBatcher:
    def __init__(self, model, num_pages, max_batch, max_blocks, max_context):
        self.max_batch, self.num_pages, self.max_blocks = max_batch, num_pages, max_blocks
        self.max_context = max_context
        self.seqs, self.queue, self.active, self.steps = {}, [], [], 0

    def submit(self, prompt, n):
        assert len(prompt) + n <= self.max_context
        sid = len(self.seqs)
        self.seqs[sid] = {"left": len(prompt) + n - 1, "p": len(prompt), "n": n, "out": 0}
        self.queue.append(sid)
        return sid

    def step(self):
        while self.queue and len(self.active) < self.max_batch:
            self.active.append(self.queue.pop(0))
        if not self.active:
            return 0
        n = len(self.active)
        for sid in list(self.active):
            s = self.seqs[sid]
            s["left"] -= 1
            done_prompt = s["p"] + s["n"] - 1 - s["left"]   # tokens fed so far
            if done_prompt >= s["p"]:
                s["out"] += 1
            if s["left"] == 0:
                self.active.remove(sid)
        self.steps += 1
        return n

    def poll(self, sid):
        s = self.seqs[sid]
        return np.zeros(s["out"], np.int32), s["left"] == 0

    def stats(self):
        return {"steps": self.steps, "preemptions": 0, "waiting": len(self.queue), "active": len(self.active),
                "free_pages": self.num_pages}

    def close(self):
        pass


class _FakeApi:
    made = {}

    @staticmethod
    def device_layer(w, kp, vp):
        return {"w": w, "k_pool": kp, "v_pool": vp}

    class Model:
        def __init__(self, cfg, layers, **kw):
            _FakeApi.made["model"] = kw

        def close(self):
            pass

    @staticmethod
    def Batcher(model, **kw):
        _FakeApi.made["batcher"] = kw
        return _FakeBatcher(model, **kw)


def test_batching_accounting():
    cfg = {"vocab": 1000, "n_kv_heads": 4, "head_dim": 128}
    t = iter(range(1000))
    res = bench.time_batching(_FakeApi, cfg, [{}, {}], None, None, None, lambda n: (n, n), lambda: None,
                              lambda: float(next(t)), n_seq=10, max_batch=4, new_tokens=5, seed=7)
    plens = bench.batching_prompts(7, 10)
    assert res["prompt_tokens"] == sum(plens)
    assert res["generated_tokens"] == 10 * 5
    assert res["token_steps"] == sum(p + 5 - 1 for p in plens)
    assert res["steps"] >= res["token_steps"] / 4 and res["mean_batch"] <= 4
    assert res["seconds"] == 1.0 and res["generated_tok_per_s"] == 50.0
    mk = _FakeApi.made
    max_ctx = max(plens) + 5
    assert mk["batcher"]["max_context"] == max_ctx == mk["model"]["max_context"]
    assert mk["batcher"]["max_blocks"] == (max_ctx + 15) // 16
    assert mk["batcher"]["num_pages"] == 4 * ((max_ctx + 15) // 16)   # every slot can reach its longest sequence


def test_batching_prompts_are_seeded_and_in_range():
    a, b = bench.batching_prompts(3, 64), bench.batching_prompts(3, 64)
    assert a == b and min(a) >= 16 and max(a) <= 128
