"""placeholder: metric formulas (full bench follows)."""


def pages_tflops(m, n, k, t_us):
    return 2.0 * m * n * k / (t_us * 1e-6) / 1e12


def pages_gbps(m, n, k, t_us):
    return (m * k + k * n + 2.0 * m * n) / (t_us * 1e-6) / 1e9
