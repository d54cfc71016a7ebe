"""Write tests/golden/tiny_oracle.txt from the fp64 oracle alone.

The fixture records the oracle's results on the tiny workload (1 sequence,
2 heads, d_k = d_v = 16, fp32 inputs from seed 1001): a 64-token prefill with
chunk 16 and a checkpoint every 32 tokens, then 8 verify steps of T = 4 with
accepted_len ~ U{0..4}.  It guards the oracle against silent change between
machines and edits: the test recomputes everything and compares.  Nothing
here comes from the CUDA path.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import kda_inputs as ki  # noqa: E402
import oracle  # noqa: E402


def tiny_run():
    w = ki.TINY
    rng = np.random.default_rng(w.seed)
    H, d = w.num_heads, w.d
    pre = ki.gen_tokens(rng, [w.extra["prefill_len"]], H, d)
    sess = oracle.OracleSession(3, H, d, d)
    o_pre, nck = sess.prefill(pre, [0], ckpt_every=w.extra["ckpt_every"],
                              ckpt_slots=np.array([[1, 2]]))
    outs, accs = [], []
    for _ in range(w.extra["steps"]):
        tok = ki.gen_tokens(rng, [w.extra["T"]], H, d)
        outs.append(sess.verify(tok, [0]))
        a = ki.accepted_uniform(rng, 1, w.extra["T"])
        accs.append(int(a[0]))
        sess.commit(a, [0])
    return o_pre, nck, sess.pool, np.stack(outs), accs


def lines():
    o_pre, nck, pool, outs, accs = tiny_run()
    out = ["# tiny workload, fp64 oracle; values printed with %.17g"]
    out.append("n_ckpt %d" % int(nck[0]))
    out.append("accepted " + " ".join(str(a) for a in accs))
    for s in range(3):
        out.append("state_slot%d_sum %.17g" % (s, pool[s].sum()))
        out.append("state_slot%d_sumsq %.17g" % (s, (pool[s] ** 2).sum()))
    out.append("prefill_out_sum %.17g" % o_pre.sum())
    out.append("prefill_out_last " + " ".join("%.17g" % x for x in o_pre[-1, 0, :4]))
    out.append("verify_out_sum %.17g" % outs.sum())
    out.append("verify_out_last " + " ".join("%.17g" % x for x in outs[-1, -1, 1, :4]))
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle.txt"), "w") as f:
        f.write("\n".join(lines()) + "\n")
    print("wrote tiny_oracle.txt")
