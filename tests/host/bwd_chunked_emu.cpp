// Host run of the chunk-form backward bodies of the library (bwd_chunked_body.cuh;
// fp32 or bf16 q, k, v, dout): one std::thread per CUDA thread of a CTA and a std::barrier for
// its x.sync(), the CTAs one after another. Reads raw float32 inputs from a
// directory and writes the gradients there. Test infrastructure: the tests
// compare its output with the gradient oracle.
#include <barrier>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>
#include "bwd_chunked_body.cuh"
using namespace gdn::cbwd;
struct HostX {
  int tid, nt;
  float* smem;
  std::barrier<>* bar;
  void sync() { bar->arrive_and_wait(); }
};
template <class F>
void run_cta(int nt, int smem_floats, F body) {
  std::vector<float> smem(smem_floats, std::nanf(""));
  std::barrier<> bar(nt);
  std::vector<std::thread> th;
  for (int t = 0; t < nt; ++t)
    th.emplace_back([&, t] { HostX x{t, nt, smem.data(), &bar}; body(x); });
  for (auto& t : th) t.join();
}
static std::vector<float> readf(const char* dir, const char* name, size_t n) {
  std::vector<float> v(n);
  char p[512];
  snprintf(p, sizeof p, "%s/%s.bin", dir, name);
  FILE* f = fopen(p, "rb");
  if (!f || fread(v.data(), 4, n, f) != n) { fprintf(stderr, "read %s\n", p); exit(1); }
  fclose(f);
  return v;
}
static void writef(const char* dir, const char* name, const std::vector<float>& v) {
  char p[512];
  snprintf(p, sizeof p, "%s/%s.bin", dir, name);
  FILE* f = fopen(p, "wb");
  fwrite(v.data(), 4, v.size(), f);
  fclose(f);
}
static std::vector<unsigned short> readh(const char* dir, const char* name, size_t n) {
  std::vector<unsigned short> v(n);
  char p[512];
  snprintf(p, sizeof p, "%s/%s.bin", dir, name);
  FILE* f = fopen(p, "rb");
  if (!f || fread(v.data(), 2, n, f) != n) { fprintf(stderr, "read %s\n", p); exit(1); }
  fclose(f);
  return v;
}
// BF: q, k, v, dout are read as bf16 bit patterns (the GPU entry point's input
// type), else as float32
template <int DK, int DV, bool BF>
int run(const char* dir, int N, int H, int T, int has_h0, int has_dhT) {
  constexpr int RB = 32, NT = 256;
  const int nch = (T + C - 1) / C;
  const size_t tok = (size_t)N * T, zc = (size_t)N * nch * H;
  std::vector<float> qf, kf, vf, of;
  std::vector<unsigned short> qh, kh, vh, oh;
  if (BF) {
    qh = readh(dir, "q", tok * H * DK); kh = readh(dir, "k", tok * H * DK);
    vh = readh(dir, "v", tok * H * DV); oh = readh(dir, "dout", tok * H * DV);
  } else {
    qf = readf(dir, "q", tok * H * DK); kf = readf(dir, "k", tok * H * DK);
    vf = readf(dir, "v", tok * H * DV); of = readf(dir, "dout", tok * H * DV);
  }
  const void* q = BF ? (const void*)qh.data() : (const void*)qf.data();
  const void* k = BF ? (const void*)kh.data() : (const void*)kf.data();
  const void* v = BF ? (const void*)vh.data() : (const void*)vf.data();
  const void* dout = BF ? (const void*)oh.data() : (const void*)of.data();
  auto g = readf(dir, "g", tok * H), beta = readf(dir, "beta", tok * H);
  std::vector<float> h0, dhT;
  if (has_h0) h0 = readf(dir, "h0", (size_t)N * H * DK * DV);
  if (has_dhT) dhT = readf(dir, "dhT", (size_t)N * H * DK * DV);
  auto ws = [&](size_t per) { return std::vector<float>(zc * per, std::nanf("")); };
  auto G = ws(C), Tm = ws(C * C), W = ws(C * DK), U0 = ws(C * DV), P = ws(C * C),
       U = ws(C * DV), S = ws(DV * DK), dSx = ws(DV * DK), dU = ws(C * DV);
  auto dOS = ws(C * DK), dKbar = ws(C * DK), dW = ws(C * DK), dKb = ws(C * DK),
       dKs = ws(C * DK), dVb = ws(C * DV), dP = ws(C * C), dT = ws(C * C),
       X = ws(C * C), dA = ws(C * C), KK = ws(C * C);
  std::vector<float> dq(tok * H * DK, NAN), dk(tok * H * DK, NAN), dv(tok * H * DV, NAN),
      dg(tok * H, NAN), dbeta(tok * H, NAN), dh0((size_t)N * H * DK * DV, NAN);
  Args a{q, k, v, dout, g.data(), beta.data(),
         has_h0 ? h0.data() : nullptr, has_dhT ? dhT.data() : nullptr, N, H, T, nch,
         G.data(), Tm.data(), W.data(), U0.data(), P.data(), U.data(), S.data(), dSx.data(), dU.data(),
         dOS.data(), dKbar.data(), dW.data(), dKb.data(), dVb.data(), dP.data(), dT.data(), X.data(),
         dA.data(), KK.data(), dKs.data(),
         dq.data(), dk.data(), dv.data(), dg.data(), dbeta.data(), dh0.data()};
  for (size_t z = 0; z < zc; ++z)
    run_cta(NT, prep_smem<DK, DV, BF>(), [&](HostX& x) { prep_body<DK, DV, BF>(x, a, (int)z); });
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h)
      for (int rb = 0; rb < DV / RB; ++rb)
        run_cta(NT, fwd_smem<DK, RB>(), [&](HostX& x) { fwd_body<DK, DV, RB, BF>(x, a, rb, h, n); });
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h)
      for (int rb = 0; rb < DV / RB; ++rb)
        run_cta(NT, rev_smem<DK, RB>(), [&](HostX& x) { rev_body<DK, DV, RB, BF>(x, a, rb, h, n); });
  for (size_t z = 0; z < zc; ++z)
    run_cta(NT, grad_smem<DK, DV, BF>(NT), [&](HostX& x) { grad_body<DK, DV, BF>(x, a, (int)z); });
  writef(dir, "dq", dq); writef(dir, "dk", dk); writef(dir, "dv", dv);
  writef(dir, "dg", dg); writef(dir, "dbeta", dbeta); writef(dir, "dh0", dh0);
  return 0;
}
template <bool BF>
int dispatch(const char* dir, int N, int H, int T, int DK, int DV, int h0, int dhT) {
  if (DK == 64 && DV == 64) return run<64, 64, BF>(dir, N, H, T, h0, dhT);
  if (DK == 128 && DV == 128) return run<128, 128, BF>(dir, N, H, T, h0, dhT);
  if (DK == 64 && DV == 128) return run<64, 128, BF>(dir, N, H, T, h0, dhT);
  if (DK == 128 && DV == 64) return run<128, 64, BF>(dir, N, H, T, h0, dhT);
  return 3;
}
int main(int argc, char** argv) {
  if (argc < 9) return 2;
  const char* dir = argv[1];
  int N = atoi(argv[2]), H = atoi(argv[3]), T = atoi(argv[4]), DK = atoi(argv[5]),
      DV = atoi(argv[6]), h0 = atoi(argv[7]), dhT = atoi(argv[8]);
  const bool bf = argc > 9 && atoi(argv[9]) != 0;
  return bf ? dispatch<true>(dir, N, H, T, DK, DV, h0, dhT)
            : dispatch<false>(dir, N, H, T, DK, DV, h0, dhT);
}
