// Host-side interfaces shared by the runtime translation units.
#pragma once

#include <cuda_runtime.h>

#include "eri_device.cuh"

struct eri_plan;

namespace eri {
namespace screen {
struct Screen;
// Builds the plan-level Schwarz screen (pair data, Q factors, per-class
// quartet sets) for eri_build_J; returns an eri_status.
int build(eri_plan* p, cudaStream_t st);
void destroy(Screen* s);
}  // namespace screen

namespace host {
int launch_class(eri_plan* p, const int l[4], EriLaunch& P, int mode, cudaStream_t st);
void canonical_order(const int l[4], int canon[4]);
bool plan_spherical(const eri_plan* p);
int plan_nshell(const eri_plan* p);
const int* plan_fo(const eri_plan* p);
const int* plan_poff(const eri_plan* p);
int plan_npmax(const eri_plan* p, int l);  // largest primitive count of the shells of l
// host copies of the caller's shell data; present only when the plan has a
// screen (schwarz_tau > 0)
const int* plan_L(const eri_plan* p);
const int* plan_nprim(const eri_plan* p);
const double* plan_centers(const eri_plan* p);
const double* plan_exps(const eri_plan* p);
const double* plan_coefs(const eri_plan* p);  // the caller's raw contraction coefficients
int plan_nsm(const eri_plan* p);
int* plan_dfo(const eri_plan* p);
screen::Screen*& plan_screen(eri_plan* p);
int class_launcher(const int l[4], int (**launch)(const EriLaunch*, int, int, int, cudaStream_t), int* slots);
void fill_plan_inputs(const eri_plan* p, EriLaunch& P);
bool plan_contracted(const eri_plan* p);
double* plan_scratch(eri_plan* p, size_t doubles, int* rc);  // grows the plan's scratch; rc = eri_status
int plan_device(const eri_plan* p);
int built_lmax();
double plan_tau(const eri_plan* p);
size_t plan_nprim_total(const eri_plan* p);
const double* plan_dcoef(const eri_plan* p);
int class_grid(const int l[4], int nsm, long long n, long long* blocks, long long* scratch);
// tier of the class's kernel: 0 register, 1 staged, 2 cooperative; -1 if not built
int class_tier(const int l[4]);
}  // namespace host
}  // namespace eri
