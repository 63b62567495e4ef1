"""The oracle's pins catch plausible mistakes: each case plants one slip in a copy of
oracle/ (CPU only) and runs tests/test_oracle_pins.py against the copy, which must fail.

The slips are the kinds a restatement of the method can make: a sign in the delta, the
decay applied after the update or not at all, the output read before the update, beta or
the output scale dropped, a wrong GQA head map, the conv taps in
reverse, SiLU without its x, the conv tail not advanced, the L2 norm without its square
root, and in the chunked form a decay exponent of the wrong sign, W h added instead of
subtracted, M without its diagonal; in the gates, logits swapped or sigmoid mirrored; in
the layer helpers, the q and k channels swapped, the v channels shifted by one head,
bf16 rounding toward zero instead of to nearest even, and the per-head (v_heads) branch
reading the wrong k-head.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

C_SRC, CHUNKED, INIT = "gdn_oracle.c", "chunked.py", "__init__.py"
MUTATIONS = {
    "delta sign": [(C_SRC, "sk[j] = b * (vt[j] - sk[j]);", "sk[j] = b * (vt[j] + sk[j]);")],
    "decay after the update": [
        (C_SRC, "        /* S <- exp(g) S */\n        for (int i = 0; i < dk * dv; ++i) h[i] *= a;\n", ""),
        (C_SRC, "        /* o_t = scale * S_t q_t */\n",
         "        for (int i = 0; i < dk * dv; ++i) h[i] *= a;\n        /* o_t = scale * S_t q_t */\n")],
    "output before the update": [
        (C_SRC, "        /* o_t = scale * S_t q_t */\n"
                "        double *ot = J->o + ((size_t)t * J->Hv + hv) * dv;\n"
                "        for (int j = 0; j < dv; ++j) {\n"
                "            double acc = 0.0;\n"
                "            for (int i = 0; i < dk; ++i) acc += h[(size_t)i * dv + j] * qn[i];\n"
                "            ot[j] = J->scale * acc;\n"
                "        }\n", ""),
        (C_SRC, "        /* S <- exp(g) S */\n",
         "        double *ot = J->o + ((size_t)t * J->Hv + hv) * dv;\n"
         "        for (int j = 0; j < dv; ++j) {\n"
         "            double acc = 0.0;\n"
         "            for (int i = 0; i < dk; ++i) acc += h[(size_t)i * dv + j] * qn[i];\n"
         "            ot[j] = J->scale * acc;\n"
         "        }\n"
         "        /* S <- exp(g) S */\n")],
    "beta dropped": [(C_SRC, "sk[j] = b * (vt[j] - sk[j]);", "sk[j] = (vt[j] - sk[j]) + 0.0 * b;")],
    "scale dropped": [(C_SRC, "ot[j] = J->scale * acc;", "ot[j] = acc;")],
    "no decay": [(C_SRC, "const double a = exp(J->g[(size_t)t * J->Hv + hv]);",
                  "const double a = 1.0 + 0.0 * J->g[(size_t)t * J->Hv + hv];")],
    "GQA head map": [(C_SRC, "const int hk = hv / (J->Hv / J->Hk);", "const int hk = hv % J->Hk;")],
    "conv taps reversed": [(C_SRC, "z += w[(size_t)c * 4 + j] * xt[t + j];",
                            "z += w[(size_t)c * 4 + j] * xt[t + 3 - j];")],
    "SiLU without x": [(C_SRC, "= z / (1.0 + exp(-z));", "= 1.0 / (1.0 + exp(-z));")],
    "conv tail not advanced": [(C_SRC, "state_out[((size_t)n * 3 + j) * C + c] = xt[L + j];",
                                "state_out[((size_t)n * 3 + j) * C + c] = xt[j];")],
    "L2 norm without sqrt": [(C_SRC, "const double inv = 1.0 / sqrt(ss + eps);",
                              "const double inv = 1.0 / (ss + eps);")],
    "chunked decay sign": [(CHUNKED, "np.exp(np.where(lower_incl, diff, 0.0))",
                            "np.exp(np.where(lower_incl, -diff, 0.0))")],
    "chunked W h sign": [(CHUNKED, "Vnew = U - W @ h0", "Vnew = U + W @ h0")],
    "chunked M without diagonal": [(CHUNKED, "Mqk = np.where(lower_incl,", "Mqk = np.where(lower_strict,")],
    "gate logits swapped": [(INIT, "return -softplus(a_raw), sigmoid(b_raw)",
                             "return -softplus(b_raw), sigmoid(a_raw)")],
    "sigmoid mirrored": [(INIT, "np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))",
                          "np.where(x >= 0, e / (1.0 + e), 1.0 / (1.0 + e))")],
    "q and k channels swapped": [
        (INIT, "q = y[:, :Hk * dk].reshape(T, Hk, dk)",
         "q = y[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk)"),
        (INIT, "k = y[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk)",
         "k = y[:, :Hk * dk].reshape(T, Hk, dk)")],
    "v channels one head late": [
        (INIT, "v = y[:, 2 * Hk * dk:2 * Hk * dk + Hv * dv].reshape(T, Hv, dv)",
         "v = np.roll(y[:, 2 * Hk * dk:2 * Hk * dk + Hv * dv], dv, axis=1).reshape(T, Hv, dv)")],
    "bf16 rounding toward zero": [
        (INIT, "    return torch.from_numpy(np.ascontiguousarray(a, np.float64)).float().to(\n"
               "        torch.bfloat16).double().numpy()",
         "    f = np.ascontiguousarray(a, np.float64).astype(np.float32)\n"
         "    return (f.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)"
         ".astype(np.float64) + 0 * torch.zeros(1).numpy()")],
    "v_heads subset with the wrong k-head": [(INIT, "        hk = hv // G\n", "        hk = hv % Hk\n")],
}


def _copy_oracle(dst, edits):
    src = os.path.join(ROOT, "oracle")
    shutil.copytree(src, os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    for name, old, new in edits:
        path = os.path.join(dst, "oracle", name)
        with open(path) as f:
            text = f.read()
        assert text.count(old) == 1, "mutation anchor not found once in %s: %r" % (name, old)
        with open(path, "w") as f:
            f.write(text.replace(old, new))


def _run_pins(dst):
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(dst), ROOT]))
    return subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q",
                           "-p", "no:cacheprovider"], cwd=str(dst), env=env,
                          capture_output=True, text=True, timeout=600)


def test_unmutated_copy_passes_and_is_the_one_imported(tmp_path):
    _copy_oracle(tmp_path, [])
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(tmp_path), ROOT]))
    where = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"],
                           cwd=str(tmp_path), env=env, capture_output=True, text=True)
    assert where.stdout.strip().startswith(str(tmp_path)), where.stdout + where.stderr
    r = _run_pins(tmp_path)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_fail_on_a_planted_mistake(tmp_path, name):
    _copy_oracle(tmp_path, MUTATIONS[name])
    r = _run_pins(tmp_path)
    # exit code 1: tests ran and at least one failed (not a collection or usage error)
    assert r.returncode == 1, "pins did not catch '%s':\n%s" % (name, r.stdout[-2000:])
